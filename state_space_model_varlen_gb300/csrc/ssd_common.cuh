// Device helpers shared by the scan kernels: the Philox4x32-10 counter-based
// generator and stochastic rounding of fp32 states to fp16 for cache writes
// (vLLM PR #61501 "Details": the stochastic-rounding Philox seed is read from
// a device buffer), and the stores of one thread's run of state values.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace ssd {

// Philox4x32 with ten rounds (Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11): words 0 and 2 of the counter are
// multiplied by the two round multipliers, the high and low halves of the
// products are mixed with words 1 and 3 and the key; the key advances by the
// two Weyl increments before every round after the first.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// The four random words of elements 4q .. 4q+3 of a tensor (stream 0: the
// state cache, 1: the per-chunk state output), seed from the caller's buffer.
__device__ __forceinline__ uint4 sr_block(uint64_t seed, uint64_t q, uint32_t stream) {
    return philox4x32_10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), stream, 0u), (uint32_t)seed,
                         (uint32_t)(seed >> 32));
}

__device__ __forceinline__ uint32_t sr_word(uint4 w, uint32_t i) {
    return i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
}

// Stochastic rounding of a float to fp16 with one random word r: with lo the
// fp16 value of v rounded toward zero and hi the next one away from zero
// (infinity above the largest finite value, whose spacing 32 is used there),
// round to hi when (|v| - |lo|) / spacing * 2^32 > r.  Every step is exact:
// |v| - |lo| holds only the bits that truncation dropped, the spacing is a power
// of two, and the comparison with the integer r is done on the rounded-up
// integer part.  Values fp16 holds exactly, infinities and NaN pass unchanged.
__device__ __forceinline__ __half sr_f16(float v, uint32_t r) {
    if (!isfinite(v)) return __float2half_rn(v);
    const float a = fabsf(v);
    const __half lo_h = __float2half_rz(a);
    const float lo = __half2float(lo_h);
    __half out = lo_h;
    if (lo != a) {
        const __half hi_h = __ushort_as_half((unsigned short)(__half_as_ushort(lo_h) + 1));
        const float spacing = (__half_as_ushort(lo_h) == 0x7BFF) ? 32.f : __half2float(hi_h) - lo;
        const unsigned long long t = __float2ull_ru(((a - lo) / spacing) * 4294967296.0f);
        if (t > (unsigned long long)r) out = hi_h;
    }
    return v < 0.f ? __hneg(out) : out;
}

// Store n consecutive state values of one thread, starting at flat element
// index e0 of the destination tensor, converting to the storage type with
// round-to-nearest-even, or (fp16 with a seed) with stochastic rounding.
template <typename StT> struct StateStore {
    __device__ static void run(StT *dst, const float *v, int n, uint64_t, const uint64_t *, uint32_t) {
        for (int j = 0; j < n; ++j) dst[j] = static_cast<StT>(v[j]);
    }
};
template <> struct StateStore<__nv_bfloat16> {
    __device__ static void run(__nv_bfloat16 *dst, const float *v, int n, uint64_t, const uint64_t *, uint32_t) {
        for (int j = 0; j < n; ++j) dst[j] = __float2bfloat16_rn(v[j]);
    }
};
template <> struct StateStore<__half> {
    __device__ static void run(__half *dst, const float *v, int n, uint64_t e0, const uint64_t *seed,
                               uint32_t stream) {
        if (seed == nullptr) {
            for (int j = 0; j < n; ++j) dst[j] = __float2half_rn(v[j]);
            return;
        }
        const uint64_t s = *seed;
        uint64_t q = ~0ull;
        uint4 w = make_uint4(0, 0, 0, 0);
        for (int j = 0; j < n; ++j) {
            const uint64_t e = e0 + (uint64_t)j;
            if ((e >> 2) != q) {
                q = e >> 2;
                w = sr_block(s, q, stream);
            }
            dst[j] = sr_f16(v[j], sr_word(w, (uint32_t)(e & 3)));
        }
    }
};

}  // namespace ssd

namespace ssd {

// Snapshot of one sequence's initial state (CTA-wide: every thread of the
// block calls it with the same s).  Multi-sequence calls keep snapshot
// semantics (vLLM PR #62922 "Details"): a sequence reads its slot as it was
// before the call even when another sequence writes that slot.  If sequence s
// has an initial state and its slot is the final slot of any other sequence,
// the slot's state_bytes are copied to states + s * state_bytes and flags[s]
// is set to 1 (else 0); the scan kernels then read the copy.
struct SnapshotArgs {
    const int32_t *slot_idx, *final_slot_idx;   // final_slot_idx NULL: slot_idx
    int64_t slot_stride, final_slot_stride;     // elements between entries (>= 1)
    const uint8_t *has_init;
    int32_t S, num_slots;
    const uint8_t *cache;                       // [num_slots, state_bytes]
    size_t state_bytes;
    int32_t *flags;                             // [S]
    uint8_t *states;                            // [S, state_bytes]
};

__device__ __forceinline__ void snapshot_sequence(const SnapshotArgs &a, int s, int *conflict_smem) {
    const bool init = a.has_init != nullptr && a.has_init[s] != 0;
    const int slot = init ? a.slot_idx[(int64_t)s * a.slot_stride] : -1;
    if (threadIdx.x == 0) *conflict_smem = 0;
    __syncthreads();
    if (init && slot >= 0 && slot < a.num_slots) {
        int c = 0;
        for (int j = threadIdx.x; j < a.S; j += blockDim.x) {
            const int f = a.final_slot_idx ? a.final_slot_idx[(int64_t)j * a.final_slot_stride]
                                           : a.slot_idx[(int64_t)j * a.slot_stride];
            c |= (j != s && f == slot);
        }
        if (c) *conflict_smem = 1;
    }
    __syncthreads();
    const int cf = *conflict_smem;
    if (threadIdx.x == 0) a.flags[s] = cf;
    if (cf) {
        const uint8_t *src = a.cache + (size_t)slot * a.state_bytes;
        uint8_t *dst = a.states + (size_t)s * a.state_bytes;
        if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | a.state_bytes) & 15u) == 0) {
            const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
            for (size_t i = threadIdx.x; i < a.state_bytes / 16; i += blockDim.x) d4[i] = s4[i];
        } else {
            for (size_t i = threadIdx.x; i < a.state_bytes; i += blockDim.x) dst[i] = src[i];
        }
    }
    __syncthreads();
}

}  // namespace ssd
