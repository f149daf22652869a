// Token-by-token SIMT scan of the Mamba2 SSD recurrence.
//
// This is the "short path" for continuations of a few tokens (MTP
// verification: one target plus draft tokens per request, vLLM PR #52928
// "Summary"), where the work is streaming the recurrent state once through
// the SM, and the general path for shapes and dtypes the chunked tensor-core
// kernel does not cover (fp32 activations, intermediate states, other
// head/state sizes).
//
// Work split: one CTA per (sequence, head, block of 16 p-rows); warp w owns
// p-rows [4w, 4w+4) of the block and each lane owns NPL consecutive state
// columns n, so the whole state slice lives in registers (4 x NPL floats per
// thread) and one token costs one warp-level reduction per p-row for y.
// Warps never synchronise with each other.  The initial state is read
// straight from the cache slot (no gather, vLLM PR #62922 "Details") and the
// final state is written back into the same slot in the cache dtype with
// round-to-nearest-even (vLLM PR #61501 "Details").
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(__half v) { return __half2float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }

// NPL consecutive elements <-> floats; one 4/8/16-byte access when `vec`.
template <typename T, int NPL>
__device__ __forceinline__ void load_n(const T *src, float (&v)[NPL], int valid, bool vec) {
    if (vec && valid >= NPL) {
        constexpr int bytes = NPL * (int)sizeof(T);
        if constexpr (bytes == 16 || bytes == 8 || bytes == 4 || bytes == 32) {
            T tmp[NPL];
            if constexpr (bytes == 32) {
                *reinterpret_cast<uint4 *>(tmp) = __ldg(reinterpret_cast<const uint4 *>(src));
                *(reinterpret_cast<uint4 *>(tmp) + 1) = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
            } else if constexpr (bytes == 16) {
                *reinterpret_cast<uint4 *>(tmp) = __ldg(reinterpret_cast<const uint4 *>(src));
            } else if constexpr (bytes == 8) {
                *reinterpret_cast<uint2 *>(tmp) = __ldg(reinterpret_cast<const uint2 *>(src));
            } else {
                *reinterpret_cast<uint32_t *>(tmp) = __ldg(reinterpret_cast<const unsigned int *>(src));
            }
#pragma unroll
            for (int j = 0; j < NPL; ++j) v[j] = to_f(tmp[j]);
            return;
        }
    }
#pragma unroll
    for (int j = 0; j < NPL; ++j) v[j] = j < valid ? to_f(src[j]) : 0.f;
}

template <typename T, int NPL>
__device__ __forceinline__ void store_n(T *dst, const float (&v)[NPL], int valid, bool vec) {
    T tmp[NPL];
#pragma unroll
    for (int j = 0; j < NPL; ++j) tmp[j] = from_f<T>(v[j]);
    if (vec && valid >= NPL) {
        constexpr int bytes = NPL * (int)sizeof(T);
        if constexpr (bytes == 32) {
            reinterpret_cast<uint4 *>(dst)[0] = reinterpret_cast<const uint4 *>(tmp)[0];
            reinterpret_cast<uint4 *>(dst)[1] = reinterpret_cast<const uint4 *>(tmp)[1];
            return;
        } else if constexpr (bytes == 16) {
            // states are written once and not read again here: streaming store
            __stcs(reinterpret_cast<uint4 *>(dst), *reinterpret_cast<const uint4 *>(tmp));
            return;
        } else if constexpr (bytes == 8) {
            *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<const uint2 *>(tmp);
            return;
        } else if constexpr (bytes == 4) {
            *reinterpret_cast<uint32_t *>(dst) = *reinterpret_cast<const uint32_t *>(tmp);
            return;
        }
    }
#pragma unroll
    for (int j = 0; j < NPL; ++j)
        if (j < valid) dst[j] = tmp[j];
}

// softplus(z) = log(1 + e^z) in the overflow-safe form max(z,0) + log1p(e^-|z|)
__device__ __forceinline__ float softplus_f(float z) {
    return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z)));
}

// kDepth: tokens of input prefetched ahead of the recurrence (a register ring;
// deeper for narrow states, where registers are cheap and the chain is short).
template <typename IoT, typename StT, int NPL, int kDepth>
__device__ __forceinline__ void recurrent_scan(const ScanArgs &a, bool vec) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int pblocks = (a.P + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t bid = blockIdx.x;
    const int pb = (int)(bid % pblocks);
    const int h = (int)((bid / pblocks) % a.H);
    const int s = (int)(bid / ((int64_t)pblocks * a.H));
    const int p0 = pb * kRowsPerCta + warp * kRowsPerWarp;
    if (p0 >= a.P) return;                                   // warp-uniform
    const int g = h / a.heads_per_group;

    // ---- sequence metadata, checked on the device (loads issued together) ----
    const int64_t t0 = a.cu_seqlens[s];
    const int64_t t1 = a.cu_seqlens[s + 1];
    const bool init = a.has_init != nullptr && a.has_init[s] != 0;
    const int slot_raw = a.slot_idx != nullptr ? a.slot_idx[s] : 0;
    if (t0 < 0 || t1 < t0 || t1 > a.T) {
        if (threadIdx.x == 0 && pb == 0 && h == 0 && a.device_status)
            atomicOr(a.device_status, SSD_DEV_BAD_SEQLENS);
        return;
    }
    const bool need_slot = init || a.write_final;
    int slot = 0;
    if (need_slot) {
        slot = slot_raw;
        if (slot < 0 || slot >= a.num_slots) {
            if (threadIdx.x == 0 && pb == 0 && h == 0 && a.device_status)
                atomicOr(a.device_status, SSD_DEV_BAD_SLOT);
            return;
        }
    }

    const int n0 = lane * NPL;
    bool row_ok[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) row_ok[i] = (p0 + i) < a.P;

    // ---- initial state (fp32 in registers) ---------------------------------
    float st[kRowsPerWarp][NPL];
    const StT *cache = static_cast<const StT *>(a.state_cache);
    const int64_t slot_base = (((int64_t)slot * a.H + h) * a.P) * a.N;
    const int nvalid = a.N - n0;           // columns of this lane inside [0, N)
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        if (init && row_ok[i]) {
            load_n<StT, NPL>(cache + slot_base + (int64_t)(p0 + i) * a.N + n0, st[i], nvalid, vec);
        } else {
#pragma unroll
            for (int j = 0; j < NPL; ++j) st[i][j] = 0.f;
        }
    }

    const IoT *X = static_cast<const IoT *>(a.x);
    const IoT *Bm = static_cast<const IoT *>(a.B);
    const IoT *Cm = static_cast<const IoT *>(a.C);
    IoT *Y = static_cast<IoT *>(a.out_y);
    StT *inter = static_cast<StT *>(a.out_intermediate);
    const float Ah = a.A[h];
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
    const float Dh = a.D ? a.D[h] : 0.f;

    if constexpr (kDepth > 1) {
        // Token inputs (dt, x, B, C) do not depend on the state: they are loaded
        // kDepth tokens ahead into a register ring, so the sequential chain waits
        // on arithmetic, not on memory latency.
        float rd[kDepth], rx[kDepth][kRowsPerWarp], rb[kDepth][NPL], rc[kDepth][NPL];
        auto fetch = [&](int u, int64_t t) {
            if (t < t1) {
                rd[u] = a.dt[t * a.H + h];
                load_n<IoT, kRowsPerWarp>(X + (t * a.H + h) * a.P + p0, rx[u], a.P - p0, vec);
                const int64_t brow = (t * a.G + g) * a.N;
                load_n<IoT, NPL>(Bm + brow + n0, rb[u], nvalid, vec);
                load_n<IoT, NPL>(Cm + brow + n0, rc[u], nvalid, vec);
            }
        };
#pragma unroll
        for (int u = 0; u < kDepth; ++u) fetch(u, t0 + u);

        for (int64_t tb = t0; tb < t1; tb += kDepth) {
            // the group's dt activations, decays and inputs, then the refill; only
            // the state update below is sequential, the rest is independent work
            float dd[kDepth], dec[kDepth], xs[kDepth][kRowsPerWarp], bs[kDepth][NPL], cs[kDepth][NPL];
#pragma unroll
            for (int u = 0; u < kDepth; ++u) {
                const float z = rd[u] + bias;
                dd[u] = a.dt_softplus ? softplus_f(z) : z;
                dec[u] = expf(dd[u] * Ah);
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i) xs[u][i] = rx[u][i];
#pragma unroll
                for (int j = 0; j < NPL; ++j) { bs[u][j] = rb[u][j]; cs[u][j] = rc[u][j]; }
            }
#pragma unroll
            for (int u = 0; u < kDepth; ++u) fetch(u, tb + kDepth + u);   // tokens of the next group
            float part[kDepth][kRowsPerWarp];
#pragma unroll
            for (int u = 0; u < kDepth; ++u) {
                const bool live = tb + u < t1;
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i) {
                    const float dx = dd[u] * xs[u][i];
                    float acc = 0.f;
#pragma unroll
                    for (int j = 0; j < NPL; ++j) {
                        if (live) st[i][j] = fmaf(dec[u], st[i][j], dx * bs[u][j]);
                        acc = fmaf(cs[u][j], st[i][j], acc);
                    }
                    part[u][i] = acc;
                }
                if (live && inter) {
                    const int64_t ibase = (((tb + u) * a.H + h) * a.P + p0) * a.N;
#pragma unroll
                    for (int i = 0; i < kRowsPerWarp; ++i)
                        if (row_ok[i]) store_n<StT, NPL>(inter + ibase + (int64_t)i * a.N + n0, st[i], nvalid, vec);
                }
            }
#pragma unroll
            for (int u = 0; u < kDepth; ++u)
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        part[u][i] += __shfl_xor_sync(0xffffffffu, part[u][i], off);
#pragma unroll
            for (int u = 0; u < kDepth; ++u) {
                if (tb + u < t1 && lane < kRowsPerWarp && row_ok[lane]) {
                    float yv = 0.f;
#pragma unroll
                    for (int i = 0; i < kRowsPerWarp; ++i)
                        if (i == lane) yv = part[u][i] + Dh * xs[u][i];
                    Y[((tb + u) * a.H + h) * a.P + p0 + lane] = from_f<IoT>(yv);
                }
            }
        }
    } else {
        // wide states: registers are scarce, plain loop (occupancy hides latency)
        for (int64_t t = t0; t < t1; ++t) {
            const float z = a.dt[t * a.H + h] + bias;
            const float d = a.dt_softplus ? softplus_f(z) : z;
            const float decay = expf(d * Ah);
            float xv[kRowsPerWarp], bv[NPL], cv[NPL];
            const int64_t xrow = (t * a.H + h) * a.P + p0;
            load_n<IoT, kRowsPerWarp>(X + xrow, xv, a.P - p0, vec);
            const int64_t brow = (t * a.G + g) * a.N;
            load_n<IoT, NPL>(Bm + brow + n0, bv, nvalid, vec);
            load_n<IoT, NPL>(Cm + brow + n0, cv, nvalid, vec);
            float part[kRowsPerWarp];
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                const float dx = d * xv[i];
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < NPL; ++j) {
                    st[i][j] = fmaf(decay, st[i][j], dx * bv[j]);
                    acc = fmaf(cv[j], st[i][j], acc);
                }
                part[i] = acc;
            }
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    part[i] += __shfl_xor_sync(0xffffffffu, part[i], off);
            if (lane < kRowsPerWarp && row_ok[lane]) {
                float yv = 0.f;
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i)
                    if (i == lane) yv = part[i] + Dh * xv[i];
                Y[xrow + lane] = from_f<IoT>(yv);
            }
            if (inter) {
                const int64_t ibase = ((t * a.H + h) * a.P + p0) * a.N;
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i)
                    if (row_ok[i]) store_n<StT, NPL>(inter + ibase + (int64_t)i * a.N + n0, st[i], nvalid, vec);
            }
        }
    }

    if (a.write_final) {
        StT *out = static_cast<StT *>(a.state_cache);
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i)
            if (row_ok[i]) store_n<StT, NPL>(out + slot_base + (int64_t)(p0 + i) * a.N + n0, st[i], nvalid, vec);
    }
}

template <typename IoT, typename StT, int NPL, int kDepth>
__global__ void __launch_bounds__(kWarps * 32) recurrent_scan_kernel(ScanArgs a, bool vec) {
    recurrent_scan<IoT, StT, NPL, kDepth>(a, vec);
}

// The plain loop with four state columns per lane (N <= 128) is latency-bound
// on its few tokens per CTA: twelve resident CTAs per SM (40 registers, a few
// spills to L1) keep more loads and stores in flight than seven CTAs of 72
// registers (MTP: -12 %).
template <typename IoT, typename StT>
__global__ void __launch_bounds__(kWarps * 32, 12) recurrent_scan_kernel_n4(ScanArgs a, bool vec) {
    recurrent_scan<IoT, StT, 4, 1>(a, vec);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename IoT, typename StT, int NPL>
cudaError_t launch_one(const ScanArgs &a, dim3 grid, dim3 block, cudaStream_t stream) {
    constexpr int kDepth = NPL <= 2 ? 4 : 1;
    // vector accesses need every row start aligned to the vector width
    const bool vec = (a.N % NPL == 0) && (a.P % kRowsPerWarp == 0) && aligned16(a.x) &&
                     aligned16(a.B) && aligned16(a.C) && aligned16(a.state_cache) &&
                     aligned16(a.out_intermediate);
    if constexpr (NPL == 4 && kDepth == 1)
        recurrent_scan_kernel_n4<IoT, StT><<<grid, block, 0, stream>>>(a, vec);
    else
        recurrent_scan_kernel<IoT, StT, NPL, kDepth><<<grid, block, 0, stream>>>(a, vec);
    return cudaGetLastError();
}

template <typename IoT, typename StT>
cudaError_t launch_npl(const ScanArgs &a, cudaStream_t stream) {
    const int pblocks = (a.P + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t blocks = (int64_t)a.S * a.H * pblocks;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)blocks), block(kWarps * 32);
    if (a.N <= 32) return launch_one<IoT, StT, 1>(a, grid, block, stream);
    if (a.N <= 64) return launch_one<IoT, StT, 2>(a, grid, block, stream);
    if (a.N <= 128) return launch_one<IoT, StT, 4>(a, grid, block, stream);
    return launch_one<IoT, StT, 8>(a, grid, block, stream);
}

template <typename IoT>
cudaError_t launch_state(const ScanArgs &a, int state_dtype, cudaStream_t stream) {
    switch (state_dtype) {
        case SSD_F32: return launch_npl<IoT, float>(a, stream);
        case SSD_BF16: return launch_npl<IoT, __nv_bfloat16>(a, stream);
        case SSD_F16: return launch_npl<IoT, __half>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_recurrent(const ScanArgs &a, int io_dtype, int state_dtype,
                             cudaStream_t stream) {
    if (io_dtype == SSD_F32) return launch_state<float>(a, state_dtype, stream);
    if (io_dtype == SSD_BF16) return launch_state<__nv_bfloat16>(a, state_dtype, stream);
    return cudaErrorInvalidValue;
}

}  // namespace ssd
