// Token-by-token SIMT scan of the Mamba2 SSD recurrence.
//
// This is the "short path" for continuations of a few tokens (MTP
// verification: one target plus draft tokens per request, vLLM PR #52928
// "Summary"), where the work is streaming the recurrent state once through
// the SM, and the general path for shapes and dtypes the chunked tensor-core
// kernel does not cover (fp32 activations, intermediate states, other
// head/state sizes).
//
// Work split: one CTA of four warps per (sequence, head, block of 4 R p-rows);
// warp w owns p-rows [Rw, Rw+R) of the block (R = 4; 8 for the plain N <= 128
// kernel, 16 for ReplaySSM) and each lane owns NPL consecutive state columns
// n, so the whole state slice lives in registers (R x NPL floats per thread).
// A token's y takes one warp-level sum per p-row; on the wide-state loop the
// R sums share their shuffles by recursive halving.
// Warps never synchronise with each other.  The initial state is read
// straight from the cache slot (no gather, vLLM PR #62922 "Details"), or from
// the snapshot the snapshot pass took when another sequence of the call writes
// that slot, and the final state is written back in the cache dtype with
// round-to-nearest-even (vLLM PR #61501 "Details") or stochastic rounding.
// Optionally the state after every token (MTP) or at every chunk boundary
// (checkpoint prefill) is written as well.
//
// The same kernel runs the ReplaySSM verification step (vLLM PR #52928
// "Summary"): before the window tokens it advances the checkpoint through the
// pending ring inputs, folds them into the checkpoint when the window would
// overflow the ring, and appends the window's inputs to the ring.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "ssd_common.cuh"
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

// Sums over the warp's 32 lanes of RPW per-lane partial values, one per p-row,
// by recursive halving: at each step a lane keeps half of its values plus its
// partner's copies of that half, so RPW values take RPW - 1 + 5 - log2(RPW)
// shuffles instead of 5 RPW.  Lane l ends with the sum of row
// rowsum_row<RPW>(l); the lanes that share a row hold the same sum.
template <int RPW>
__device__ __forceinline__ float warp_rowsums(float (&v)[RPW], int lane) {
    static_assert(RPW >= 1 && RPW <= 32 && (RPW & (RPW - 1)) == 0, "power of two rows");
#pragma unroll
    for (int half = RPW / 2, off = 16; half >= 1; half /= 2, off /= 2) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float r = v[0];
#pragma unroll
    for (int off = 32 / RPW / 2; off > 0; off /= 2) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}
template <int RPW>
__device__ __forceinline__ int rowsum_row(int lane) {
    int r = 0;
#pragma unroll
    for (int half = RPW / 2, off = 16; half >= 1; half /= 2, off /= 2)
        if (lane & off) r += half;
    return r;
}
// the first lane of each group that warp_rowsums leaves holding one row's sum
template <int RPW>
__device__ __forceinline__ bool rowsum_writer(int lane) { return (lane & (32 / RPW - 1)) == 0; }

// kDepth: tokens whose y reductions are batched on the staged narrow-state path
// (kDepth > 1: inputs staged through shared memory a chunk at a time); 1 for
// wide states (plain loop, occupancy hides the loads).
// kFull: the optional parts of a call (separate final slots, strided slot
// indices, snapshot reads, per-chunk states, stochastic rounding, the
// ReplaySSM ring) are compiled in; calls without them run the plain variant,
// whose register budget they would otherwise take.
template <typename IoT, typename StT, int NPL, int kDepth, bool kFull, int RPW = 4>
__device__ __forceinline__ void recurrent_scan(const ScanArgs &a, bool vec) {
    constexpr int kRowsPerWarp = RPW;                   // p-rows of a warp
    constexpr int kRowsPerCta = kWarps * RPW;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int pblocks = (a.P + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t bid = blockIdx.x;
    const int pb = (int)(bid % pblocks);
    const int h = (int)((bid / pblocks) % a.H);
    const int s = (int)(bid / ((int64_t)pblocks * a.H));
    const int p0 = pb * kRowsPerCta + warp * kRowsPerWarp;
    // warps without rows of their own leave early, except where every warp
    // loads inputs for the CTA and meets at barriers (the staged narrow-state
    // path, the ReplaySSM prologue)
    if (kDepth == 1 && p0 >= a.P && !(kFull && a.ring_x != nullptr)) return;
    const int g = h / a.heads_per_group;

    // ---- sequence metadata, checked on the device (loads issued together) ----
    const bool replay = kFull && a.ring_x != nullptr;
    const bool reporter = threadIdx.x == 0 && pb == 0 && h == 0;
    const int64_t t0 = a.cu_seqlens[s];
    const int64_t t1 = a.cu_seqlens[s + 1];
    const bool init = replay || (a.has_init != nullptr && a.has_init[s] != 0);
    const int64_t sstride = kFull && a.slot_stride ? a.slot_stride : 1;
    const int slot_raw = a.slot_idx != nullptr ? a.slot_idx[s * sstride] : 0;
    const int fslot_raw = (kFull && a.write_final && a.final_slot_idx != nullptr)
                              ? a.final_slot_idx[s * (a.final_slot_stride ? a.final_slot_stride : 1)]
                              : slot_raw;
    if (t0 < 0 || t1 < t0 || t1 > a.T) {
        if (reporter && a.device_status) atomicOr(a.device_status, SSD_DEV_BAD_SEQLENS);
        return;
    }
    int slot = 0, fslot = 0;
    if ((init && (slot_raw < 0 || slot_raw >= a.num_slots)) ||
        (a.write_final && (fslot_raw < 0 || fslot_raw >= a.num_slots))) {
        if (reporter && a.device_status) atomicOr(a.device_status, SSD_DEV_BAD_SLOT);
        return;
    }
    if (init) slot = slot_raw;
    if (a.write_final) fslot = fslot_raw;
    // per-chunk states: rows cu_chunks[s] .. cu_chunks[s+1]-1
    StT *chunks = kFull ? static_cast<StT *>(a.out_chunk_states) : nullptr;
    int64_t crow0 = 0;
    if (chunks) {
        const int64_t c0 = a.cu_chunks[s], c1 = a.cu_chunks[s + 1];
        const int64_t nch = (t1 - t0 + a.chunk_size - 1) / a.chunk_size;
        if (c0 < 0 || c1 - c0 != nch || c1 > a.num_chunk_rows) {
            if (reporter && a.device_status) atomicOr(a.device_status, SSD_DEV_BAD_CHUNKS);
            chunks = nullptr;
        }
        crow0 = c0;
    }
    // ReplaySSM: pending ring inputs and where the window goes
    int32_t rcount = 0, rstart = 0, wpos0 = 0;
    bool fold = false;
    if (replay) {
        rcount = a.ring_count[s];
        rstart = a.ring_start[s];
        const int64_t K = t1 - t0;
        if (rcount < 0 || rcount > a.ring_window || rstart < 0 || rstart >= a.ring_capacity ||
            K > (int64_t)a.ring_capacity - a.ring_window) {
            if (reporter && a.device_status) atomicOr(a.device_status, SSD_DEV_BAD_RING);
            return;
        }
        fold = rcount + K > a.ring_window;
        wpos0 = (rstart + rcount) % a.ring_capacity;
        if (reporter) {
            a.ring_start_out[s] = fold ? wpos0 : rstart;
            a.ring_count_out[s] = fold ? 0 : rcount;
        }
    }

    const int n0 = lane * NPL;
    bool row_ok[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) row_ok[i] = (p0 + i) < a.P;

    // ---- initial state (fp32 in registers) ---------------------------------
    float st[kRowsPerWarp][NPL];
    const int64_t head_off = ((int64_t)h * a.P) * a.N;
    const int64_t slot_base = (int64_t)slot * a.H * a.P * a.N + head_off;
    const int64_t fslot_base = (int64_t)fslot * a.H * a.P * a.N + head_off;
    const StT *src = static_cast<const StT *>(a.state_cache) + slot_base;
    if (kFull && a.snap_flag != nullptr && a.snap_flag[s] != 0)
        src = static_cast<const StT *>(a.snap_states) + (int64_t)s * a.H * a.P * a.N + head_off;
    const int nvalid = a.N - n0;           // columns of this lane inside [0, N)
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        if (init && row_ok[i]) {
            load_n<StT, NPL>(src + (int64_t)(p0 + i) * a.N + n0, st[i], nvalid, vec);
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
    const int nw = nvalid < NPL ? (nvalid > 0 ? nvalid : 0) : NPL;
    // this warp's rows of the state (cache dtype; stochastic rounding for fp16
    // with a seed), at flat element index base of a [rows, H, P, N] tensor
    auto store_rows = [&](StT *dst, int64_t base, uint32_t stream) {
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            if (!row_ok[i] || nw == 0) continue;
            const int64_t e = base + (int64_t)(p0 + i) * a.N + n0;
            if constexpr (kFull && std::is_same<StT, __half>::value) {
                if (a.sr_seed != nullptr) {
                    StateStore<StT>::run(dst + e, st[i], nw, (uint64_t)e, a.sr_seed, stream);
                    continue;
                }
            }
            store_n<StT, NPL>(dst + e, st[i], nvalid, vec);
        }
    };
    // the state after token t, when t ends a chunk of its sequence
    auto chunk_store = [&](int64_t t) {
        const int64_t pos = t - t0;
        if (chunks && ((pos + 1) % a.chunk_size == 0 || t == t1 - 1))
            store_rows(chunks, ((crow0 + pos / a.chunk_size) * a.H) * a.P * a.N + head_off, 1u);
    };
    // ReplaySSM: the window token t goes to ring position wpos0 + (t - t0)
    auto ring_store = [&](int64_t t) {
        if (!replay) return;
        int64_t pos = wpos0 + (t - t0);             // < 2 capacity: wpos0 < capacity, K <= capacity
        if (pos >= a.ring_capacity) pos -= a.ring_capacity;
        const int64_t rrow = (int64_t)slot * a.ring_capacity + pos;
        if (lane < kRowsPerWarp && p0 + lane < a.P)
            static_cast<IoT *>(a.ring_x)[(rrow * a.H + h) * a.P + p0 + lane] = X[(t * a.H + h) * a.P + p0 + lane];
        if (pb == 0 && warp == 0) {
            if (lane == 0) a.ring_dt[rrow * a.H + h] = a.dt[t * a.H + h];
            if (h % a.heads_per_group == 0)
                for (int j = 0; j < NPL; ++j)
                    if (n0 + j < a.N)
                        static_cast<IoT *>(a.ring_B)[(rrow * a.G + g) * a.N + n0 + j] =
                            Bm[(t * a.G + g) * a.N + n0 + j];
        }
    };
    // one token of the recurrence for this warp's rows, with y and the
    // optional per-token, per-chunk and ring writes
    auto step = [&](int64_t t, float d, float decay, const float (&xv)[kRowsPerWarp],
                    const float (&bv)[NPL], const float (&cv)[NPL]) {
        const int64_t xrow = (t * a.H + h) * a.P + p0;
        float part[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const float dx = d * xv[i];
            float acc = lane == 0 ? Dh * xv[i] : 0.f;      // D x enters the row sum once
#pragma unroll
            for (int j = 0; j < NPL; ++j) {
                st[i][j] = fmaf(decay, st[i][j], dx * bv[j]);
                acc = fmaf(cv[j], st[i][j], acc);
            }
            part[i] = acc;
        }
        {
            const float yv = warp_rowsums<kRowsPerWarp>(part, lane);
            const int r = rowsum_row<kRowsPerWarp>(lane);
            if (rowsum_writer<kRowsPerWarp>(lane) && p0 + r < a.P) Y[xrow + r] = from_f<IoT>(yv);
        }
        if (inter) {
            const int64_t ibase = ((t * a.H + h) * a.P + p0) * a.N;
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i)
                if (row_ok[i]) store_n<StT, NPL>(inter + ibase + (int64_t)i * a.N + n0, st[i], nvalid, vec);
        }
        chunk_store(t);
        ring_store(t);
    };
    // Wide states (N = 128) with eight or sixteen rows a warp: the tokens'
    // inputs are staged through shared memory with asynchronous copies, up to
    // kTs tokens in one memory round trip with no register staging, then run
    // in order.  For ReplaySSM the pending ring tokens come first and advance
    // the checkpoint (folded into the cache when the window overflows the
    // ring), then the window tokens produce y; for MTP it is the window alone.
    bool unified = false;
    if constexpr (kDepth == 1 && NPL == 4 && RPW >= 8) {
        if (a.N == 32 * NPL && a.P % kRowsPerCta == 0 && vec) {
            unified = true;
            constexpr int kTs = 16;
            constexpr int kNM = 32 * NPL;
            constexpr int kThr = kWarps * 32;
            constexpr int kCx = kRowsPerCta * (int)sizeof(IoT) / 16;   // 16-byte chunks of a token's x
            constexpr int kCb = kNM * (int)sizeof(IoT) / 16;           // ... of its B (and C) row
            __shared__ __align__(16) IoT u_x[kTs][kRowsPerCta];
            __shared__ __align__(16) IoT u_b[kTs][kNM];
            __shared__ __align__(16) IoT u_c[kTs][kNM];
            __shared__ __align__(16) float u_dt[kTs];
            __shared__ float u_d[kTs], u_dec[kTs];
            const int tid = threadIdx.x, xr0 = warp * kRowsPerWarp, pc0 = pb * kRowsPerCta;
            const IoT *RX = static_cast<const IoT *>(a.ring_x);
            const IoT *RB = static_cast<const IoT *>(a.ring_B);
            const int32_t ntot = rcount + (int32_t)(t1 - t0);
            auto rrow = [&](int32_t j) {                // j < window <= capacity, rstart < capacity
                int32_t q = rstart + j;
                if (q >= a.ring_capacity) q -= a.ring_capacity;
                return (int64_t)slot * a.ring_capacity + q;
            };
            auto cp16 = [](void *dst, const void *src) {
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                             "l"(src) : "memory");
            };
            if (fold && rcount == 0) store_rows(static_cast<StT *>(a.state_cache), slot_base, 0u);
            for (int32_t j0 = 0; j0 < ntot; j0 += kTs) {
                const int nj = ntot - j0 < kTs ? ntot - j0 : kTs;
                for (int e = tid; e < nj * (kCx + 2 * kCb); e += kThr) {
                    const int jj = e / (kCx + 2 * kCb), c = e % (kCx + 2 * kCb), j = j0 + jj;
                    const bool ring = j < rcount;
                    if (c < kCx) {
                        const IoT *src = (ring ? RX + (rrow(j) * a.H + h) * a.P
                                               : X + ((t0 + j - rcount) * a.H + h) * a.P) + pc0;
                        cp16(&u_x[jj][c * 16 / (int)sizeof(IoT)], src + c * 16 / (int)sizeof(IoT));
                    } else if (c < kCx + kCb) {
                        const int cb = c - kCx;
                        const IoT *src = ring ? RB + (rrow(j) * a.G + g) * a.N
                                              : Bm + ((t0 + j - rcount) * a.G + g) * a.N;
                        cp16(&u_b[jj][cb * 16 / (int)sizeof(IoT)], src + cb * 16 / (int)sizeof(IoT));
                    } else if (!ring) {
                        const int cc = c - kCx - kCb;
                        cp16(&u_c[jj][cc * 16 / (int)sizeof(IoT)],
                             Cm + ((t0 + j - rcount) * a.G + g) * a.N + cc * 16 / (int)sizeof(IoT));
                    }
                }
                if (tid < nj) {
                    const int j = j0 + tid;
                    u_dt[tid] = j < rcount ? a.ring_dt[rrow(j) * a.H + h] : a.dt[(t0 + j - rcount) * a.H + h];
                }
                asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
                __syncthreads();
                if (tid < nj) {                             // once per CTA, not per warp
                    const float z = u_dt[tid] + bias;
                    const float d = a.dt_softplus ? softplus_f(z) : z;
                    u_d[tid] = d;
                    u_dec[tid] = expf(d * Ah);
                }
                __syncthreads();
                for (int jj = 0; jj < nj; ++jj) {
                    const int j = j0 + jj;
                    const float d = u_d[jj], decay = u_dec[jj];
                    if (j < rcount) {
#pragma unroll
                        for (int i = 0; i < kRowsPerWarp; ++i) {
                            const float dx = d * to_f(u_x[jj][xr0 + i]);
#pragma unroll
                            for (int q = 0; q < NPL; ++q) st[i][q] = fmaf(decay, st[i][q], dx * to_f(u_b[jj][n0 + q]));
                        }
                        if (j == rcount - 1 && fold) store_rows(static_cast<StT *>(a.state_cache), slot_base, 0u);
                    } else {
                        float xv[kRowsPerWarp], bv[NPL], cv[NPL];
#pragma unroll
                        for (int i = 0; i < kRowsPerWarp; ++i) xv[i] = to_f(u_x[jj][xr0 + i]);
#pragma unroll
                        for (int q = 0; q < NPL; ++q) {
                            bv[q] = to_f(u_b[jj][n0 + q]);
                            cv[q] = to_f(u_c[jj][n0 + q]);
                        }
                        step(t0 + j - rcount, d, decay, xv, bv, cv);
                    }
                }
                __syncthreads();
            }
        }
    }
    if (replay && !unified) {
        // advance the checkpoint through the pending ring inputs (no output):
        // the CTA loads kRs tokens' inputs at a time into shared memory
        // together, every load in flight at once, then each warp replays them
        // for its rows
        constexpr int kRs = 8;
        constexpr int kNM = 32 * NPL;
        constexpr int kThr = kWarps * 32;
        __shared__ float rs_d[kRs], rs_dec[kRs];   // dt' and exp(dt' A) of each staged token
        __shared__ float rs_x[kRs][kRowsPerCta];
        __shared__ __align__(16) float rs_b[kRs][kNM];
        const int tid = threadIdx.x, pc0 = pb * kRowsPerCta, xr0 = warp * kRowsPerWarp;
        const IoT *RX = static_cast<const IoT *>(a.ring_x);
        const IoT *RB = static_cast<const IoT *>(a.ring_B);
        auto rrow = [&](int32_t j) {                // j < window <= capacity, rstart < capacity
            int32_t q = rstart + j;
            if (q >= a.ring_capacity) q -= a.ring_capacity;
            return (int64_t)slot * a.ring_capacity + q;
        };
        for (int32_t j0 = 0; j0 < rcount; j0 += kRs) {
            const int nj = rcount - j0 < kRs ? rcount - j0 : kRs;
            float vx[kRs * kRowsPerCta / kThr > 0 ? kRs * kRowsPerCta / kThr : 1];
            float vb[kRs * kNM / kThr];
            float vd = 0.f;
            if (tid < nj) vd = a.ring_dt[rrow(j0 + tid) * a.H + h];
#pragma unroll
            for (int k = 0; k < kRs * kRowsPerCta / kThr; ++k) {
                const int e = tid + k * kThr, jj = e / kRowsPerCta, r = e % kRowsPerCta;
                vx[k] = (jj < nj && pc0 + r < a.P) ? to_f(RX[(rrow(j0 + jj) * a.H + h) * a.P + pc0 + r]) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < kRs * kNM / kThr; ++k) {
                const int e = tid + k * kThr, jj = e / kNM, n = e % kNM;
                vb[k] = (jj < nj && n < a.N) ? to_f(RB[(rrow(j0 + jj) * a.G + g) * a.N + n]) : 0.f;
            }
            if (tid < kRs) {                            // once per CTA, not per warp
                const float z = vd + bias;
                const float d = a.dt_softplus ? softplus_f(z) : z;
                rs_d[tid] = d;
                rs_dec[tid] = expf(d * Ah);
            }
#pragma unroll
            for (int k = 0; k < kRs * kRowsPerCta / kThr; ++k) {
                const int e = tid + k * kThr;
                rs_x[e / kRowsPerCta][e % kRowsPerCta] = vx[k];
            }
#pragma unroll
            for (int k = 0; k < kRs * kNM / kThr; ++k) {
                const int e = tid + k * kThr;
                rs_b[e / kNM][e % kNM] = vb[k];
            }
            __syncthreads();
            for (int jj = 0; jj < nj; ++jj) {
                const float d = rs_d[jj], decay = rs_dec[jj];
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i) {
                    const float dx = d * rs_x[jj][xr0 + i];
#pragma unroll
                    for (int j = 0; j < NPL; ++j) st[i][j] = fmaf(decay, st[i][j], dx * rs_b[jj][n0 + j]);
                }
            }
            __syncthreads();
        }
        if (fold) store_rows(static_cast<StT *>(a.state_cache), slot_base, 0u);
    }

    if constexpr (kDepth > 1) {
        // Narrow states (N <= 64): a token's state update is a few FMAs, so its
        // inputs would dominate if each token's loads were waited for one by one.
        // All four warps load the inputs (dt, x of the CTA's 16 rows, B, C) of
        // kStage tokens at a time into shared memory together -- the next chunk
        // is loaded into registers while the current one is computed and stored
        // behind it -- and each warp runs its rows' recurrence out of shared
        // memory, kDepth tokens at a time with their y reductions batched.
        constexpr int kStage = 32;
        constexpr int kNMax = 32 * NPL;
        constexpr int kThr = kWarps * 32;
        constexpr int kXe = kStage * kRowsPerCta / kThr;        // x elements per thread
        constexpr int kBe = kStage * kNMax / kThr;              // B (and C) elements per thread
        static_assert(kStage % kDepth == 0 && kStage <= kThr, "chunk layout");
        __shared__ float s_dt[2][kStage];
        __shared__ float s_x[2][kStage][kRowsPerCta];
        __shared__ __align__(16) float s_b[2][kStage][kNMax];
        __shared__ __align__(16) float s_c[2][kStage][kNMax];
        const int tid = threadIdx.x;
        const int pc0 = pb * kRowsPerCta;                       // first row of the CTA
        float rdt, rx[kXe], rb[kBe], rc[kBe];
        auto fetch = [&](int64_t tb) {                          // global -> registers
            const int64_t td = tb + tid;
            rdt = (tid < kStage && td < t1) ? a.dt[td * a.H + h] : 0.f;
#pragma unroll
            for (int k = 0; k < kXe; ++k) {
                const int e = tid + k * kThr, tt = e / kRowsPerCta, r = e % kRowsPerCta;
                const int64_t t = tb + tt;
                rx[k] = (t < t1 && pc0 + r < a.P) ? to_f(X[(t * a.H + h) * a.P + pc0 + r]) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < kBe; ++k) {
                const int e = tid + k * kThr, tt = e / kNMax, n = e % kNMax;
                const int64_t t = tb + tt;
                const bool v = t < t1 && n < a.N;
                rb[k] = v ? to_f(Bm[(t * a.G + g) * a.N + n]) : 0.f;
                rc[k] = v ? to_f(Cm[(t * a.G + g) * a.N + n]) : 0.f;
            }
        };
        auto put = [&](int buf) {                               // registers -> shared memory
            if (tid < kStage) s_dt[buf][tid] = rdt;
#pragma unroll
            for (int k = 0; k < kXe; ++k) {
                const int e = tid + k * kThr;
                s_x[buf][e / kRowsPerCta][e % kRowsPerCta] = rx[k];
            }
#pragma unroll
            for (int k = 0; k < kBe; ++k) {
                const int e = tid + k * kThr;
                s_b[buf][e / kNMax][e % kNMax] = rb[k];
                s_c[buf][e / kNMax][e % kNMax] = rc[k];
            }
        };
        const int xr0 = warp * kRowsPerWarp;                    // this warp's rows within the CTA's
        fetch(t0);
        put(0);
        __syncthreads();
        int buf = 0;
        for (int64_t cb = t0; cb < t1; cb += kStage) {
            const bool more = cb + kStage < t1;
            if (more) fetch(cb + kStage);                       // next chunk, in flight meanwhile
#pragma unroll 1
            for (int ub = 0; ub < kStage; ub += kDepth) {
                const int64_t tb = cb + ub;
                if (tb >= t1) break;
                float dd[kDepth], dec[kDepth], xs[kDepth][kRowsPerWarp];
#pragma unroll
                for (int u = 0; u < kDepth; ++u) {
                    const float z = s_dt[buf][ub + u] + bias;
                    dd[u] = a.dt_softplus ? softplus_f(z) : z;
                    dec[u] = expf(dd[u] * Ah);
#pragma unroll
                    for (int i = 0; i < kRowsPerWarp; ++i) xs[u][i] = s_x[buf][ub + u][xr0 + i];
                }
                float part[kDepth * kRowsPerWarp];            // [token u][row i] at u R + i
#pragma unroll
                for (int u = 0; u < kDepth; ++u) {
                    const bool live = tb + u < t1;
                    float bs[NPL], cs[NPL];
#pragma unroll
                    for (int j = 0; j < NPL; ++j) {
                        bs[j] = s_b[buf][ub + u][n0 + j];
                        cs[j] = s_c[buf][ub + u][n0 + j];
                    }
#pragma unroll
                    for (int i = 0; i < kRowsPerWarp; ++i) {
                        const float dx = dd[u] * xs[u][i];
                        float acc = lane == 0 ? Dh * xs[u][i] : 0.f;   // D x enters the row sum once
#pragma unroll
                        for (int j = 0; j < NPL; ++j) {
                            if (live) st[i][j] = fmaf(dec[u], st[i][j], dx * bs[j]);
                            acc = fmaf(cs[j], st[i][j], acc);
                        }
                        part[u * kRowsPerWarp + i] = acc;
                    }
                    if (live && inter) {
                        const int64_t ibase = (((tb + u) * a.H + h) * a.P + p0) * a.N;
#pragma unroll
                        for (int i = 0; i < kRowsPerWarp; ++i)
                            if (row_ok[i]) store_n<StT, NPL>(inter + ibase + (int64_t)i * a.N + n0, st[i], nvalid, vec);
                    }
                    if (live) {
                        chunk_store(tb + u);
                        ring_store(tb + u);
                    }
                }
                {
                    // the kDepth x R row sums share their shuffles (recursive halving)
                    constexpr int kSums = kDepth * kRowsPerWarp;
                    const float yv = warp_rowsums<kSums>(part, lane);
                    const int r = rowsum_row<kSums>(lane), u = r / kRowsPerWarp, i = r % kRowsPerWarp;
                    if (rowsum_writer<kSums>(lane) && tb + u < t1 && p0 + i < a.P)
                        Y[((tb + u) * a.H + h) * a.P + p0 + i] = from_f<IoT>(yv);
                }
            }
            if (more) put(buf ^ 1);
            __syncthreads();                                    // every warp is done with buf
            buf ^= 1;
        }
    } else {
        // wide states: registers are scarce, plain loop (occupancy hides latency)
        bool staged = unified;
        if constexpr (kFull) {
            if (replay && !unified) {
                // ReplaySSM window: its tokens' inputs staged through shared
                // memory kWs tokens at a time, every load in flight together
                // (the window's first chunk alongside nothing else to wait for)
                staged = true;
                constexpr int kWs = 8;
                constexpr int kNM = 32 * NPL;
                constexpr int kThr = kWarps * 32;
                constexpr int kXe = kWs * kRowsPerCta / kThr > 0 ? kWs * kRowsPerCta / kThr : 1;
                __shared__ float ws_d[kWs], ws_dec[kWs];
                __shared__ float ws_x[kWs][kRowsPerCta];
                __shared__ __align__(16) float ws_b[kWs][kNM];
                __shared__ __align__(16) float ws_c[kWs][kNM];
                const int tid = threadIdx.x, pc0 = pb * kRowsPerCta, xr0 = warp * kRowsPerWarp;
                for (int64_t tb = t0; tb < t1; tb += kWs) {
                    const int nj = t1 - tb < kWs ? (int)(t1 - tb) : kWs;
                    float vx[kXe], vb[kWs * kNM / kThr], vc[kWs * kNM / kThr];
                    float vd = 0.f;
                    if (tid < nj) vd = a.dt[(tb + tid) * a.H + h];
#pragma unroll
                    for (int k = 0; k < kXe; ++k) {
                        const int e = tid + k * kThr, jj = e / kRowsPerCta, r = e % kRowsPerCta;
                        vx[k] = (jj < nj && pc0 + r < a.P) ? to_f(X[((tb + jj) * a.H + h) * a.P + pc0 + r]) : 0.f;
                    }
#pragma unroll
                    for (int k = 0; k < kWs * kNM / kThr; ++k) {
                        const int e = tid + k * kThr, jj = e / kNM, n = e % kNM;
                        const bool v = jj < nj && n < a.N;
                        const int64_t row = ((tb + jj) * a.G + g) * a.N + n;
                        vb[k] = v ? to_f(Bm[row]) : 0.f;
                        vc[k] = v ? to_f(Cm[row]) : 0.f;
                    }
                    if (tid < kWs) {                            // once per CTA, not per warp
                        const float z = vd + bias;
                        const float d = a.dt_softplus ? softplus_f(z) : z;
                        ws_d[tid] = d;
                        ws_dec[tid] = expf(d * Ah);
                    }
#pragma unroll
                    for (int k = 0; k < kXe; ++k) {
                        const int e = tid + k * kThr;
                        if (e < kWs * kRowsPerCta) ws_x[e / kRowsPerCta][e % kRowsPerCta] = vx[k];
                    }
#pragma unroll
                    for (int k = 0; k < kWs * kNM / kThr; ++k) {
                        const int e = tid + k * kThr;
                        ws_b[e / kNM][e % kNM] = vb[k];
                        ws_c[e / kNM][e % kNM] = vc[k];
                    }
                    __syncthreads();
                    for (int jj = 0; jj < nj; ++jj) {
                        float xv[kRowsPerWarp], bv[NPL], cv[NPL];
#pragma unroll
                        for (int i = 0; i < kRowsPerWarp; ++i) xv[i] = ws_x[jj][xr0 + i];
#pragma unroll
                        for (int j = 0; j < NPL; ++j) {
                            bv[j] = ws_b[jj][n0 + j];
                            cv[j] = ws_c[jj][n0 + j];
                        }
                        step(tb + jj, ws_d[jj], ws_dec[jj], xv, bv, cv);
                    }
                    __syncthreads();
                }
            }
        }
        if (!staged) {
            for (int64_t t = t0; t < t1; ++t) {
                const float z = a.dt[t * a.H + h] + bias;
                const float d = a.dt_softplus ? softplus_f(z) : z;
                const float decay = expf(d * Ah);
                float xv[kRowsPerWarp], bv[NPL], cv[NPL];
                load_n<IoT, kRowsPerWarp>(X + (t * a.H + h) * a.P + p0, xv, a.P - p0, vec);
                const int64_t brow = (t * a.G + g) * a.N;
                load_n<IoT, NPL>(Bm + brow + n0, bv, nvalid, vec);
                load_n<IoT, NPL>(Cm + brow + n0, cv, nvalid, vec);
                step(t, d, decay, xv, bv, cv);
            }
        }
    }

    if (a.write_final) store_rows(static_cast<StT *>(a.state_cache), fslot_base, 0u);
}

template <typename IoT, typename StT, int NPL, int kDepth, bool kFull>
__global__ void __launch_bounds__(kWarps * 32) recurrent_scan_kernel(ScanArgs a, bool vec) {
    recurrent_scan<IoT, StT, NPL, kDepth, kFull>(a, vec);
}

// The plain loop with four state columns per lane (N <= 128) streams its
// states (MTP: the state after every token): eight p-rows a warp and eight
// resident CTAs per SM (64 registers, a few spills to L1) keep more state
// stores in flight per warp than four rows at twelve CTAs (MTP: -9 %), and
// share each token's dt', decay and B, C loads over twice the rows.
template <typename IoT, typename StT>
__global__ void __launch_bounds__(kWarps * 32, 8) recurrent_scan_kernel_n4(ScanArgs a, bool vec) {
    recurrent_scan<IoT, StT, 4, 1, false, 8>(a, vec);
}

// ReplaySSM verification: sixteen p-rows a warp (all 64 rows of a head in one
// CTA), so that the ring staging, each token's dt' and decay, and the
// metadata are shared by four times as many rows.
template <typename IoT, typename StT>
__global__ void __launch_bounds__(kWarps * 32, 4) recurrent_replay_kernel_n4(ScanArgs a, bool vec) {
    recurrent_scan<IoT, StT, 4, 1, true, 16>(a, vec);
}

// The same shape with the optional parts (ReplaySSM, final slots, ...): eight
// resident CTAs per SM, so the replay prologue's memory latency overlaps.
template <typename IoT, typename StT>
__global__ void __launch_bounds__(kWarps * 32, 8) recurrent_scan_kernel_n4_full(ScanArgs a, bool vec) {
    recurrent_scan<IoT, StT, 4, 1, true>(a, vec);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether a call uses any optional part (then the kFull variant runs).
bool uses_options(const ScanArgs &a) {
    return a.final_slot_idx != nullptr || (a.slot_stride != 0 && a.slot_stride != 1) ||
           a.snap_flag != nullptr || a.out_chunk_states != nullptr || a.sr_seed != nullptr ||
           a.ring_x != nullptr;
}

// vector accesses need every row start aligned to the vector width
bool vec_ok(const ScanArgs &a, int npl, int rows_per_warp) {
    return (a.N % npl == 0) && (a.P % rows_per_warp == 0) && aligned16(a.x) && aligned16(a.B) &&
           aligned16(a.C) && aligned16(a.state_cache) && aligned16(a.out_intermediate) &&
           aligned16(a.out_chunk_states) && aligned16(a.snap_states) && aligned16(a.ring_x) &&
           aligned16(a.ring_B);
}

template <typename IoT, typename StT, int NPL>
cudaError_t launch_one(const ScanArgs &a, dim3 grid, dim3 block, cudaStream_t stream) {
    constexpr int kDepth = NPL <= 2 ? 4 : 1;
    const bool vec = vec_ok(a, NPL, kRowsPerWarp);
    if (uses_options(a)) {
        if constexpr (NPL == 4 && kDepth == 1)
            recurrent_scan_kernel_n4_full<IoT, StT><<<grid, block, 0, stream>>>(a, vec);
        else
            recurrent_scan_kernel<IoT, StT, NPL, kDepth, true><<<grid, block, 0, stream>>>(a, vec);
    }
    else if constexpr (NPL == 4 && kDepth == 1) {
        constexpr int kRows = kWarps * 8;                   // p-rows of a CTA of this kernel
        const int64_t nb = (int64_t)a.S * a.H * ((a.P + kRows - 1) / kRows);
        if (nb > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        recurrent_scan_kernel_n4<IoT, StT><<<(unsigned)nb, block, 0, stream>>>(a, vec_ok(a, 4, 8));
    } else
        recurrent_scan_kernel<IoT, StT, NPL, kDepth, false><<<grid, block, 0, stream>>>(a, vec);
    return cudaGetLastError();
}

template <typename IoT, typename StT>
cudaError_t launch_npl(const ScanArgs &a, cudaStream_t stream) {
    const int pblocks = (a.P + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t blocks = (int64_t)a.S * a.H * pblocks;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)blocks), block(kWarps * 32);
    if (a.ring_x != nullptr && a.N > 64 && a.N <= 128) {
        // ReplaySSM verification: one CTA per (sequence, head, 64 p-rows)
        constexpr int kRows = kWarps * 16;
        const int64_t rblocks = (int64_t)a.S * a.H * ((a.P + kRows - 1) / kRows);
        if (rblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        recurrent_replay_kernel_n4<IoT, StT><<<(unsigned)rblocks, block, 0, stream>>>(a, vec_ok(a, 4, 16));
        return cudaGetLastError();
    }
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
