// Chunked SSD scan on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// The pages run Mamba2's prefill scan as five Triton launches -- cumsum,
// chunk state, state passing, bmm, chunk scan -- or as FlashInfer's fused
// two-launch scan over packed cu_seqlens with the chunk metadata derived on
// the device (vLLM PR #61501 "Details"); the initial state is read straight
// from the cache slot and each chunk's entering state is kept on chip rather
// than gathered into a dense buffer (vLLM PR #62922 "Details").  This file is
// a single-pass design of the same computation for one GB300 SM:
//
// Launch 1 (prep): sort the sequences by block count, longest first, into the
//   workspace (the only scratch memory), so the persistent CTAs below take
//   the long chains first.
// Launch 2 (scan): one persistent CTA per SM.  A work item is one sequence and
//   two heads of the same B/C group; its tokens are walked in 128-token blocks
//   and the recurrent state h [2 heads x 64 x 128] never leaves the SM (fp32 in
//   registers).  Per block, with cum_t = sum_{r<=t} dt'_r A (within the block):
//     G   = C B^T                         tcgen05, K = n, fp32 in TMEM
//     S_h = G o exp(cum_t - cum_s) dt'_s  (s <= t), bf16, written back in TMEM
//     Y   = C h^T                         tcgen05 (state entering the block)
//     Y  *= exp(cum_t)                    per row and head, in TMEM
//     Y  += S_h X_h                       tcgen05, A operand from TMEM
//     y   = Y + D x                       bf16, TMA store
//     Sc  = Xw^T B,  Xw = exp(cum_end - cum_s) dt'_s x_s split into bf16 hi+lo
//     h   = exp(cum_end) h + Sc           fp32, written to the cache slot at the end
//   The hi/lo split keeps the state contributions accurate to ~2^-16 so final
//   states meet fp32-storage accuracy; everything else runs on bf16 operands
//   with fp32 accumulation.
//
// Warp roles (16 warps): warp 0 TMA producer, warp 1 MMA issuer, warp 2 TMEM
// owner, warps 4-7 "token" warpgroup (dt softplus + cumsum, S, row scaling,
// epilogue; lane = token), warps 8-15 "state" warpgroups (Xw^T, state update,
// cache I/O; lane = head x p, each warpgroup one half of the 128 state columns).
// All hand-offs are mbarriers; every wait is bounded and sets an abort flag
// plus SSD_DEV_TIMEOUT in device_status instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "sm100.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kQ = 128;            // tokens per block
constexpr int kP = 64;             // head dim
constexpr int kN = 128;            // state dim
constexpr int kSlots = 5;          // TMA ring of 32 KB tiles (B, C, X per block)
constexpr int kTileBytes = 32768;
constexpr int kHalfBytes = 16384;
constexpr int kThreads = 512;
constexpr uint64_t kSpinLimit = 4000000000ull;   // clock cycles (~2 s) per wait

// TMEM columns
constexpr uint32_t kColG = 0;      // G / S (in place), lanes = tokens
constexpr uint32_t kColY = 128;    // Y, lanes = tokens, cols = head x p
constexpr uint32_t kColSc = 256;   // state contributions, lanes = head x p, cols = n
constexpr uint32_t kColXhi = 384;  // Xw^T hi, lanes = head x p, cols = s/2
constexpr uint32_t kColXlo = 448;  // Xw^T lo

constexpr uint32_t kIdG = idesc_bf16(128, 128, false, false);    // C . B^T
constexpr uint32_t kIdY = idesc_bf16(128, 128, false, false);    // C . h^T
constexpr uint32_t kIdSX = idesc_bf16(128, 64, false, true);     // S_h . X_h
constexpr uint32_t kIdSc = idesc_bf16(128, 128, false, true);    // Xw^T . B

struct Params {
    int64_t T;
    int32_t S, H, G, hpg, num_items, num_slots;
    int32_t dt_softplus, write_final, state_dtype;
    const float *dt, *dt_bias, *A, *D;
    const int32_t *cu_seqlens, *slot_idx, *order;
    const uint8_t *has_init;
    void *state_cache, *out_y;
    int32_t *device_status;
};

struct __align__(1024) Smem {
    uint8_t slot[kSlots][kTileBytes];     // TMA ring
    uint8_t hbuf[2][kHalfBytes];          // h (bf16) K-major: [n half][row = head*64+p][128 B]
    float cum[2][2][kQ];                  // [array buffer][head][token]
    float dtp[2][2][kQ];                  // dt'
    float vfac[2][2][kQ];                 // exp(cum_{end of 32-block} - cum_s) dt'_s
    float wfac[2][2][kQ];                 // exp(cum_end - cum_s) dt'_s
    float cumE[2][2][4];                  // cum at the end of each 32-token block
    float wtot[2][2][4];                  // scan scratch [buffer][head][warp]
    uint64_t full[kSlots], empty[kSlots];
    uint64_t scan_bar[2], dt_ready[2], arrays_free[2];
    uint64_t g_ready, s_ready, hs_ready, yinter_ready, y_scaled, y_ready, y_free, ytile;
    uint64_t xp_ready, sc_ready, sc_free, drain;
    uint32_t tmem_base;
    int32_t abort_flag;
};

// ---------------------------------------------------------------------------
// work enumeration, identical in every role
// ---------------------------------------------------------------------------
struct Chunk {
    int32_t seq, h0, g, slot;
    int64_t row0;        // first token of this block
    int32_t l;           // valid tokens in this block
    bool init, first, last, empty_item;
};

struct Walker {
    const Params *p;
    int cta, grid;
    int round = 0;
    // current item
    bool have = false;
    int32_t seq = 0, h0 = 0, g = 0, slot = 0, len = 0, nb = 0, b = 0;
    int64_t t0 = 0;
    bool init = false;

    __device__ Walker(const Params *pp) : p(pp), cta(blockIdx.x), grid(gridDim.x) {}

    // Load the next valid item; returns false when this CTA has no more work.
    __device__ bool next_item(bool report) {
        const int hp_per_seq = p->H / 2;
        while (true) {
            const int64_t base = (int64_t)round * grid;
            const int64_t idx = base + ((round & 1) ? (grid - 1 - cta) : cta);
            ++round;
            if (base >= p->num_items) return false;
            if (idx >= p->num_items) continue;
            const int rank = (int)(idx / hp_per_seq);
            const int hp = (int)(idx % hp_per_seq);
            seq = p->order[rank];
            h0 = hp * 2;
            g = h0 / p->hpg;
            const int64_t a = p->cu_seqlens[seq], e = p->cu_seqlens[seq + 1];
            if (a < 0 || e < a || e > p->T) {
                if (report && p->device_status) atomicOr(p->device_status, SSD_DEV_BAD_SEQLENS);
                continue;
            }
            init = p->has_init != nullptr && p->has_init[seq] != 0;
            slot = 0;
            if (init || p->write_final) {
                slot = p->slot_idx[seq];
                if (slot < 0 || slot >= p->num_slots) {
                    if (report && p->device_status) atomicOr(p->device_status, SSD_DEV_BAD_SLOT);
                    continue;
                }
            }
            t0 = a;
            len = (int32_t)(e - a);
            nb = (len + kQ - 1) / kQ;
            b = 0;
            return true;
        }
    }

    // Next event: a block of an item, or (if want_empty) an item without tokens.
    __device__ bool next(Chunk &c, bool want_empty, bool report = false) {
        while (true) {
            if (!have || b >= nb) {
                if (!next_item(report)) return false;
                have = true;
                if (nb == 0) {
                    b = 0;
                    if (want_empty) {
                        c.seq = seq; c.h0 = h0; c.g = g; c.slot = slot; c.row0 = t0; c.l = 0;
                        c.init = init; c.first = c.last = true; c.empty_item = true;
                        return true;
                    }
                    continue;
                }
            }
            c.seq = seq; c.h0 = h0; c.g = g; c.slot = slot; c.init = init;
            c.row0 = t0 + (int64_t)b * kQ;
            c.l = min(kQ, len - b * kQ);
            c.first = (b == 0);
            c.last = (b == nb - 1);
            c.empty_item = false;
            ++b;
            return true;
        }
    }
};

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
// Single-thread wait (producer / MMA issuer).
__device__ __forceinline__ bool wait_bar(Smem &sm, uint64_t *bar, uint32_t parity,
                                         int32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t_start = clock64();
    uint32_t it = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++it & 255u) == 0) {
            if (*(volatile int32_t *)&sm.abort_flag) return false;
            if (clock64() - t_start > kSpinLimit) {
                atomicExch(&sm.abort_flag, 1);
                if (status) atomicOr(status, SSD_DEV_TIMEOUT);
                return false;
            }
        }
    }
    return true;
}

// Whole-warp wait with a warp-uniform result (all 32 lanes must call it).
// A barrier phase never runs two completions ahead of its slowest waiter in
// this kernel, so once one lane observes completion every lane will.
__device__ __forceinline__ bool warp_wait(Smem &sm, uint64_t *bar, uint32_t parity,
                                          int32_t *status) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const uint64_t t_start = clock64();
    uint32_t it = 0;
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if ((++it & 255u) == 0) {
            int give_up = 0;
            if ((threadIdx.x & 31) == 0) {
                if (*(volatile int32_t *)&sm.abort_flag) {
                    give_up = 1;
                } else if (clock64() - t_start > kSpinLimit) {
                    atomicExch(&sm.abort_flag, 1);
                    if (status) atomicOr(status, SSD_DEV_TIMEOUT);
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
    }
}

__device__ __forceinline__ float softplus_f(float z) {
    return fmaxf(z, 0.f) + log1pf(__expf(-fabsf(z)));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename StT> __device__ __forceinline__ void load_state_row(const StT *src, float (&h)[64]);
template <> __device__ __forceinline__ void load_state_row<float>(const float *src, float (&h)[64]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(src) + i);
        h[4 * i] = v.x; h[4 * i + 1] = v.y; h[4 * i + 2] = v.z; h[4 * i + 3] = v.w;
    }
}
template <> __device__ __forceinline__ void load_state_row<__nv_bfloat16>(const __nv_bfloat16 *src, float (&h)[64]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src) + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) { h[8 * i + 2 * q] = bf16_lo(w[q]); h[8 * i + 2 * q + 1] = bf16_hi(w[q]); }
    }
}
template <> __device__ __forceinline__ void load_state_row<__half>(const __half *src, float (&h)[64]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src) + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __half2 hh = *reinterpret_cast<const __half2 *>(&w[q]);
            const float2 f = __half22float2(hh);
            h[8 * i + 2 * q] = f.x; h[8 * i + 2 * q + 1] = f.y;
        }
    }
}

template <typename StT> __device__ __forceinline__ void store_state_row(StT *dst, const float (&h)[64]);
template <> __device__ __forceinline__ void store_state_row<float>(float *dst, const float (&h)[64]) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
        reinterpret_cast<float4 *>(dst)[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
}
template <> __device__ __forceinline__ void store_state_row<__nv_bfloat16>(__nv_bfloat16 *dst, const float (&h)[64]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint4 v;
        v.x = pack_bf16(h[8 * i], h[8 * i + 1]);
        v.y = pack_bf16(h[8 * i + 2], h[8 * i + 3]);
        v.z = pack_bf16(h[8 * i + 4], h[8 * i + 5]);
        v.w = pack_bf16(h[8 * i + 6], h[8 * i + 7]);
        reinterpret_cast<uint4 *>(dst)[i] = v;
    }
}
template <> __device__ __forceinline__ void store_state_row<__half>(__half *dst, const float (&h)[64]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __half2 hh = __floats2half2_rn(h[8 * i + 2 * q], h[8 * i + 2 * q + 1]);
            w[q] = *reinterpret_cast<const uint32_t *>(&hh);
        }
        reinterpret_cast<uint4 *>(dst)[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// bf16 copy of this thread's 64 state columns into its K-major hbuf row.
__device__ __forceinline__ void write_hbuf_row(uint8_t *row, int r, const float (&h)[64]) {
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
        uint4 v;
        v.x = pack_bf16(h[8 * cc + 0], h[8 * cc + 1]);
        v.y = pack_bf16(h[8 * cc + 2], h[8 * cc + 3]);
        v.z = pack_bf16(h[8 * cc + 4], h[8 * cc + 5]);
        v.w = pack_bf16(h[8 * cc + 6], h[8 * cc + 7]);
        *reinterpret_cast<uint4 *>(row + ((cc ^ (r & 7)) << 4)) = v;
    }
}

// ---------------------------------------------------------------------------
// launch 1: longest-first order of the sequences
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 1024;
constexpr int kSortMax = 8192;

__global__ void __launch_bounds__(kPrepThreads) prep_order_kernel(const int32_t *cu, int S, int64_t T,
                                                                    int32_t *order) {
    __shared__ int32_t nb[kSortMax];
    if (S > kSortMax) {
        for (int s = threadIdx.x; s < S; s += blockDim.x) order[s] = s;
        return;
    }
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const int64_t a = cu[s], e = cu[s + 1];
        nb[s] = (a < 0 || e < a || e > T) ? 0 : (int32_t)((e - a + kQ - 1) / kQ);
    }
    __syncthreads();
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const int32_t v = nb[s];
        int rank = 0;
        for (int q = 0; q < S; ++q) {
            const int32_t u = nb[q];
            rank += (u > v) || (u == v && q < s);
        }
        order[rank] = s;
    }
}

// ---------------------------------------------------------------------------
// launch 2: the scan
// ---------------------------------------------------------------------------
template <typename StT>
__global__ void __launch_bounds__(kThreads, 1)
chunked_scan_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CUtensorMap map_y,
                    const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) { mbar_init(&sm.full[i], 1); mbar_init(&sm.empty[i], 2); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.scan_bar[i], 4);
            mbar_init(&sm.dt_ready[i], 4);
            mbar_init(&sm.arrays_free[i], 12);
        }
        mbar_init(&sm.g_ready, 1);
        mbar_init(&sm.s_ready, 4);
        mbar_init(&sm.hs_ready, 8);
        mbar_init(&sm.yinter_ready, 1);
        mbar_init(&sm.y_scaled, 4);
        mbar_init(&sm.y_ready, 1);
        mbar_init(&sm.y_free, 4);
        mbar_init(&sm.ytile, 4);
        mbar_init(&sm.xp_ready, 8);
        mbar_init(&sm.sc_ready, 1);
        mbar_init(&sm.sc_free, 8);
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    int32_t *status = p.device_status;

    if (warp == 0) {
        // ===================== TMA producer =====================
        if (lane == 0) {
            tma_prefetch_desc(&map_x);
            tma_prefetch_desc(&map_b);
            tma_prefetch_desc(&map_c);
            tma_prefetch_desc(&map_y);
            Walker wk(&p);
            Chunk c;
            uint32_t kc = 0, issued = 0;
            bool ok = true;
            while (ok && wk.next(c, false, true)) {
                const int32_t row = (int32_t)c.row0;
                for (int j = 0; j < 3; ++j) {
                    const uint32_t tile = 3 * kc + j, slot = tile % kSlots, use = tile / kSlots;
                    if (use > 0 && !(ok = wait_bar(sm, &sm.empty[slot], (use - 1) & 1, status))) break;
                    mbar_arrive_expect_tx(&sm.full[slot], kTileBytes);
                    uint8_t *dst = sm.slot[slot];
                    const CUtensorMap *m = (j == 0) ? &map_b : (j == 1) ? &map_c : &map_x;
                    const int32_t c0 = (j == 2) ? c.h0 * kP : c.g * kN;
                    const int32_t c1 = (j == 2) ? (c.h0 + 1) * kP : c.g * kN + 64;
                    tma_load_2d(dst, m, &sm.full[slot], c0, row);
                    tma_load_2d(dst + kHalfBytes, m, &sm.full[slot], c1, row);
                    issued = tile + 1;
                }
                ++kc;
            }
            // every issued load must have landed before the CTA exits
            for (uint32_t t = (issued > (uint32_t)kSlots ? issued - kSlots : 0); t < issued; ++t)
                wait_bar(sm, &sm.full[t % kSlots], (t / kSlots) & 1, nullptr);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (lane == 0) {
            Walker wk(&p);
            Chunk c;
            uint32_t kc = 0;
            bool ok = true;
            while (ok && wk.next(c, false)) {
                const uint32_t tb = 3 * kc, tcc = 3 * kc + 1, tx = 3 * kc + 2;
                const uint32_t bB = smem_u32(sm.slot[tb % kSlots]);
                const uint32_t bC = smem_u32(sm.slot[tcc % kSlots]);
                const uint32_t bX = smem_u32(sm.slot[tx % kSlots]);
                // ---- G = C B^T ----
                if (!(ok = wait_bar(sm, &sm.full[tb % kSlots], (tb / kSlots) & 1, status) &&
                           wait_bar(sm, &sm.full[tcc % kSlots], (tcc / kSlots) & 1, status)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
                    mma_ss(tmem + kColG, smem_desc_sw128(bC + off, 16, 1024),
                           smem_desc_sw128(bB + off, 16, 1024), kIdG, ks > 0);
                }
                mma_commit(&sm.g_ready);
                // ---- Y = C h^T ----
                if (!(ok = wait_bar(sm, &sm.hs_ready, kc & 1, status) &&
                           (kc == 0 || wait_bar(sm, &sm.y_free, (kc - 1) & 1, status))))
                    break;
                tc_fence_after();
                const uint32_t bH = smem_u32(sm.hbuf[0]);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
                    mma_ss(tmem + kColY, smem_desc_sw128(bC + off, 16, 1024),
                           smem_desc_sw128(bH + off, 16, 1024), kIdY, ks > 0);
                }
                mma_commit(&sm.yinter_ready);
                mma_commit(&sm.empty[tcc % kSlots]);
                mma_commit(&sm.empty[tcc % kSlots]);
                // ---- Sc = Xw^T B (hi + lo) ----
                if (!(ok = wait_bar(sm, &sm.xp_ready, kc & 1, status) &&
                           (kc == 0 || wait_bar(sm, &sm.sc_free, (kc - 1) & 1, status))))
                    break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 16; ++ks) {
                    const uint32_t acol = (ks < 8 ? kColXhi : kColXlo) + 8 * (ks & 7);
                    mma_ts(tmem + kColSc, tmem + acol,
                           smem_desc_sw128(bB + (ks & 7) * 2048, kHalfBytes, 1024), kIdSc, ks > 0);
                }
                mma_commit(&sm.sc_ready);
                mma_commit(&sm.empty[tb % kSlots]);
                mma_commit(&sm.empty[tb % kSlots]);
                // ---- Y += S_h X_h ----
                if (!(ok = wait_bar(sm, &sm.full[tx % kSlots], (tx / kSlots) & 1, status) &&
                           wait_bar(sm, &sm.s_ready, kc & 1, status) &&
                           wait_bar(sm, &sm.y_scaled, kc & 1, status)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t acol = kColG + 32 * (ks >> 1) + 16 * hh + 8 * (ks & 1);
                        mma_ts(tmem + kColY + 64 * hh, tmem + acol,
                               smem_desc_sw128(bX + hh * kHalfBytes + ks * 2048, 1024, 1024), kIdSX, 1);
                    }
                }
                mma_commit(&sm.y_ready);
                mma_commit(&sm.empty[tx % kSlots]);
                ++kc;
            }
            // drain the tensor pipe before TMEM is released
            mma_commit(&sm.drain);
            wait_bar(sm, &sm.drain, 0, nullptr);
        }
    } else if (warp >= 4 && warp < 8) {
        // ===================== token warpgroup =====================
        const int q = warp - 4;                 // lane quarter
        const int t = q * 32 + lane;            // token row within the block
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        Walker wk(&p);
        Chunk cur, nxt;
        bool have_cur = wk.next(cur, false);
        bool have_nxt = have_cur && wk.next(nxt, false);
        uint32_t kc = 0;
        bool ok = true;

        // dt softplus + within-block cumsum of dt' A for block k -> array buffer k % 2
        auto dtprep = [&](const Chunk &c, uint32_t k) -> bool {
            const int ab = k & 1;
            if (k >= 2 && !warp_wait(sm, &sm.arrays_free[ab], ((k >> 1) - 1) & 1, status)) return false;
            const bool valid = t < c.l;
            float d[2] = {0.f, 0.f}, a[2] = {0.f, 0.f};
            if (valid) {
                const float2 raw = *reinterpret_cast<const float2 *>(p.dt + (c.row0 + t) * p.H + c.h0);
                const float rv[2] = {raw.x, raw.y};
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float z = rv[hh] + (p.dt_bias ? p.dt_bias[c.h0 + hh] : 0.f);
                    d[hh] = p.dt_softplus ? softplus_f(z) : z;
                    a[hh] = d[hh] * p.A[c.h0 + hh];
                }
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float v = __shfl_up_sync(0xffffffffu, a[hh], off);
                    if (lane >= off) a[hh] += v;
                }
                if (lane == 31) sm.wtot[ab][hh][q] = a[hh];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.scan_bar[ab]);
            if (!warp_wait(sm, &sm.scan_bar[ab], (k >> 1) & 1, status)) return false;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float w0 = sm.wtot[ab][hh][0], w1 = sm.wtot[ab][hh][1];
                const float w2 = sm.wtot[ab][hh][2], w3 = sm.wtot[ab][hh][3];
                const float e0 = w0, e1 = w0 + w1, e2 = e1 + w2, e3 = e2 + w3;
                const float pre = (q == 0) ? 0.f : (q == 1) ? e0 : (q == 2) ? e1 : e2;
                const float cblk = (q == 0) ? e0 : (q == 1) ? e1 : (q == 2) ? e2 : e3;
                const float cum = a[hh] + pre;
                sm.cum[ab][hh][t] = cum;
                sm.dtp[ab][hh][t] = d[hh];
                sm.vfac[ab][hh][t] = valid ? __expf(cblk - cum) * d[hh] : 0.f;
                sm.wfac[ab][hh][t] = valid ? __expf(e3 - cum) * d[hh] : 0.f;
                if (t == 0) {
                    sm.cumE[ab][hh][0] = e0; sm.cumE[ab][hh][1] = e1;
                    sm.cumE[ab][hh][2] = e2; sm.cumE[ab][hh][3] = e3;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.dt_ready[ab]);
            return true;
        };

        if (have_cur) ok = dtprep(cur, 0);
        while (ok && have_cur) {
            const int ab = kc & 1;
            const int slotX = (3 * kc + 2) % kSlots;
            const float Dv[2] = {p.D ? p.D[cur.h0] : 0.f, p.D ? p.D[cur.h0 + 1] : 0.f};
            // ---- S_h from G, in place ----
            if (!(ok = warp_wait(sm, &sm.dt_ready[ab], (kc >> 1) & 1, status) &&
                       warp_wait(sm, &sm.g_ready, kc & 1, status)))
                break;
            tc_fence_after();
            const float cum_t[2] = {sm.cum[ab][0][t], sm.cum[ab][1][t]};
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t out0[16], out1[16];
                if (j > q) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) { out0[i] = 0u; out1[i] = 0u; }
                } else {
                    uint32_t g[32];
                    tmem_ld32(tmem + lane_off + kColG + 32 * j, g);
                    tmem_wait_ld();
                    if (j < q) {
                        const float u0 = __expf(cum_t[0] - sm.cumE[ab][0][j]);
                        const float u1 = __expf(cum_t[1] - sm.cumE[ab][1][j]);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int s = 32 * j + 2 * i;
                            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                            out0[i] = pack_bf16(g0 * u0 * sm.vfac[ab][0][s], g1 * u0 * sm.vfac[ab][0][s + 1]);
                            out1[i] = pack_bf16(g0 * u1 * sm.vfac[ab][1][s], g1 * u1 * sm.vfac[ab][1][s + 1]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int s = 32 * j + 2 * i;
                            float r0[2], r1[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float gv = __uint_as_float(g[2 * i + e]);
                                const bool keep = (s + e) <= t;
                                r0[e] = keep ? gv * (__expf(cum_t[0] - sm.cum[ab][0][s + e]) * sm.dtp[ab][0][s + e]) : 0.f;
                                r1[e] = keep ? gv * (__expf(cum_t[1] - sm.cum[ab][1][s + e]) * sm.dtp[ab][1][s + e]) : 0.f;
                            }
                            out0[i] = pack_bf16(r0[0], r0[1]);
                            out1[i] = pack_bf16(r1[0], r1[1]);
                        }
                    }
                }
                tmem_st16(tmem + lane_off + kColG + 32 * j, out0);
                tmem_st16(tmem + lane_off + kColG + 32 * j + 16, out1);
            }
            const float ecum[2] = {__expf(cum_t[0]), __expf(cum_t[1])};
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.s_ready);
                mbar_arrive(&sm.arrays_free[ab]);
            }
            // ---- dt prep of the next block (overlaps the MMAs of this one) ----
            if (have_nxt && !(ok = dtprep(nxt, kc + 1))) break;
            // ---- Y *= exp(cum_t) ----
            if (!(ok = warp_wait(sm, &sm.yinter_ready, kc & 1, status))) break;
            tc_fence_after();
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + kColY + 32 * j, r);
                tmem_wait_ld();
                const float e = ecum[j >> 1];
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * e);
                tmem_st32(tmem + lane_off + kColY + 32 * j, r);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.y_scaled);
            // ---- epilogue: y = Y + D x, in place over the X tile ----
            if (!(ok = warp_wait(sm, &sm.y_ready, kc & 1, status))) break;
            tc_fence_after();
            uint8_t *xt = sm.slot[slotX];
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + kColY + 32 * j, r);
                tmem_wait_ld();
                if (j == 3) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.y_free);
                }
                const int hh = j >> 1;
                uint8_t *row = xt + hh * kHalfBytes + t * 128;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int chunk = (j & 1) * 4 + cc;            // 8 p-values per 16-B chunk
                    uint4 *ptr = reinterpret_cast<uint4 *>(row + ((chunk ^ (t & 7)) << 4));
                    const uint4 xv = *ptr;
                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                    uint32_t yw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float y0 = __uint_as_float(r[cc * 8 + 2 * e]) + Dv[hh] * bf16_lo(xw[e]);
                        const float y1 = __uint_as_float(r[cc * 8 + 2 * e + 1]) + Dv[hh] * bf16_hi(xw[e]);
                        yw[e] = pack_bf16(y0, y1);
                    }
                    *ptr = make_uint4(yw[0], yw[1], yw[2], yw[3]);
                }
            }
            if (cur.l < kQ && t < cur.l) {
                // partial block: this row straight to global (a TMA box would overrun
                // into the next sequence)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint8_t *row = xt + hh * kHalfBytes + t * 128;
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out_y) +
                                                          (cur.row0 + t) * p.H * kP + (cur.h0 + hh) * kP);
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc)
                        dst[cc] = *reinterpret_cast<const uint4 *>(row + ((cc ^ (t & 7)) << 4));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.ytile);
            if (q == 0) {
                if (!(ok = warp_wait(sm, &sm.ytile, kc & 1, status))) break;
                if (lane == 0) {
                    if (cur.l == kQ) {
                        const int32_t row = (int32_t)cur.row0;
                        asm volatile(
                            "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                                reinterpret_cast<uint64_t>(&map_y)),
                            "r"(cur.h0 * kP), "r"(row), "r"(smem_u32(xt))
                            : "memory");
                        asm volatile(
                            "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                                reinterpret_cast<uint64_t>(&map_y)),
                            "r"((cur.h0 + 1) * kP), "r"(row), "r"(smem_u32(xt + kHalfBytes))
                            : "memory");
                        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    }
                    mbar_arrive(&sm.empty[slotX]);
                }
                __syncwarp();
            }
            cur = nxt;
            have_cur = have_nxt;
            if (have_cur) have_nxt = wk.next(nxt, false);
            ++kc;
        }
        if (q == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    } else if (warp >= 8) {
        // ===================== state warpgroups =====================
        const int wg = (warp - 8) >> 2;          // n half: columns [64 wg, 64 wg + 64)
        const int q = warp & 3;
        const int r = q * 32 + lane;             // head * 64 + p
        const int hh = r >> 6, pp = r & 63;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        Walker wk(&p);
        Chunk c;
        uint32_t kc = 0;
        bool ok = true;
        float h[64];
        StT *cache = static_cast<StT *>(p.state_cache);
        uint8_t *hrow = sm.hbuf[wg] + r * 128;
        while (ok && wk.next(c, true)) {
            const int64_t srow = ((int64_t)c.slot * p.H + c.h0 + hh) * (kP * kN) + pp * kN + wg * 64;
            if (c.first) {
                if (c.init) {
                    load_state_row<StT>(cache + srow, h);
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i) h[i] = 0.f;
                }
            }
            if (c.empty_item) {
                if (p.write_final) store_state_row<StT>(cache + srow, h);
                continue;
            }
            if (c.first) {
                // state entering block 0 of the item -> hbuf for Y = C h^T
                if (kc > 0 && !(ok = warp_wait(sm, &sm.yinter_ready, (kc - 1) & 1, status))) break;
                write_hbuf_row(hrow, r, h);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.hs_ready);
            }
            // ---- Xw^T (hi, lo) of this block into TMEM ----
            const int ab = kc & 1;
            const uint32_t tx = 3 * kc + 2;
            if (!(ok = warp_wait(sm, &sm.full[tx % kSlots], (tx / kSlots) & 1, status) &&
                       warp_wait(sm, &sm.dt_ready[ab], (kc >> 1) & 1, status) &&
                       (kc == 0 || warp_wait(sm, &sm.sc_ready, (kc - 1) & 1, status))))
                break;
            tc_fence_after();
            {
                const uint8_t *xt = sm.slot[tx % kSlots] + hh * kHalfBytes;
                const int chunk = pp >> 3, within = (pp & 7) * 2;
#pragma unroll 1
                for (int grp = 0; grp < 4; ++grp) {
                    uint32_t whi[8], wlo[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float v[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int s = wg * 64 + grp * 16 + 2 * i + e;
                            const uint16_t xb = *reinterpret_cast<const uint16_t *>(
                                xt + s * 128 + ((chunk ^ (s & 7)) << 4) + within);
                            const float wv = sm.wfac[ab][hh][s];
                            v[e] = (wv != 0.f) ? wv * __uint_as_float((uint32_t)xb << 16) : 0.f;
                        }
                        whi[i] = pack_bf16(v[0], v[1]);
                        wlo[i] = pack_bf16(v[0] - bf16_lo(whi[i]), v[1] - bf16_hi(whi[i]));
                    }
                    const uint32_t col = wg * 32 + grp * 8;
                    tmem_st8(tmem + lane_off + kColXhi + col, whi);
                    tmem_st8(tmem + lane_off + kColXlo + col, wlo);
                }
            }
            const float delta = sm.cumE[ab][hh][3];
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.xp_ready);
                mbar_arrive(&sm.arrays_free[ab]);
            }
            // ---- state update: h = exp(cum_end) h + Sc ----
            if (!(ok = warp_wait(sm, &sm.sc_ready, kc & 1, status))) break;
            tc_fence_after();
            {
                uint32_t s0[32], s1[32];
                tmem_ld32(tmem + lane_off + kColSc + wg * 64, s0);
                tmem_ld32(tmem + lane_off + kColSc + wg * 64 + 32, s1);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.sc_free);
                const float dec = __expf(delta);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    h[i] = fmaf(dec, h[i], __uint_as_float(s0[i]));
                    h[32 + i] = fmaf(dec, h[32 + i], __uint_as_float(s1[i]));
                }
            }
            if (c.last) {
                if (p.write_final) store_state_row<StT>(cache + srow, h);
            } else {
                if (!(ok = warp_wait(sm, &sm.yinter_ready, kc & 1, status))) break;
                write_hbuf_row(hrow, r, h);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.hs_ready);
            }
            ++kc;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// 2-D bf16 view [rows, inner] with 128-byte-swizzled 64 x 128 boxes.
bool make_map(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {64, kQ};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int sms = 0;
    bool attr_set[3] = {false, false, false};
};
DeviceInfo g_dev[64];
std::mutex g_dev_mu;

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

template <typename StT>
cudaError_t launch_typed(const ScanArgs &a, int st_idx, void *workspace, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        DeviceInfo &di = g_dev[dev];
        if (di.sms == 0) {
            e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
        }
        if (!di.attr_set[st_idx]) {
            e = cudaFuncSetAttribute(chunked_scan_kernel<StT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
            if (e != cudaSuccess) return e;
            di.attr_set[st_idx] = true;
        }
        sms = di.sms;
    }
    CUtensorMap mx, mb, mc, my;
    if (!make_map(&mx, a.x, (uint64_t)a.H * kP, (uint64_t)a.T) ||
        !make_map(&my, a.out_y, (uint64_t)a.H * kP, (uint64_t)a.T) ||
        !make_map(&mb, a.B, (uint64_t)a.G * kN, (uint64_t)a.T) ||
        !make_map(&mc, a.C, (uint64_t)a.G * kN, (uint64_t)a.T))
        return cudaErrorInvalidValue;
    int32_t *order = static_cast<int32_t *>(workspace);
    prep_order_kernel<<<1, kPrepThreads, 0, stream>>>(a.cu_seqlens, a.S, a.T, order);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    Params p;
    p.T = a.T;
    p.S = a.S;
    p.H = a.H;
    p.G = a.G;
    p.hpg = a.heads_per_group;
    p.num_items = a.S * (a.H / 2);
    p.num_slots = a.num_slots;
    p.dt_softplus = a.dt_softplus;
    p.write_final = a.write_final;
    p.state_dtype = st_idx;
    p.dt = a.dt;
    p.dt_bias = a.dt_bias;
    p.A = a.A;
    p.D = a.D;
    p.cu_seqlens = a.cu_seqlens;
    p.slot_idx = a.slot_idx;
    p.order = order;
    p.has_init = a.has_init;
    p.state_cache = a.state_cache;
    p.out_y = a.out_y;
    p.device_status = a.device_status;
    const int grid = p.num_items < sms ? p.num_items : sms;
    chunked_scan_kernel<StT><<<grid, kThreads, kSmemBytes, stream>>>(mx, mb, mc, my, p);
    return cudaGetLastError();
}

}  // namespace

bool chunked_supported(const ssd_scan_params &p) {
    if (p.io_dtype != SSD_BF16 || p.headdim != kP || p.dstate != kN) return false;
    if (p.nheads % 2 != 0 || (p.nheads / p.ngroups) % 2 != 0) return false;
    if (p.total_tokens >= (1LL << 31) - kQ) return false;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.B) |
                          reinterpret_cast<uintptr_t>(p.C) | reinterpret_cast<uintptr_t>(p.out_y) |
                          reinterpret_cast<uintptr_t>(p.dt) | reinterpret_cast<uintptr_t>(p.state_cache);
    if (mis & 15u) return false;
    if (p.total_tokens > 0 && encode_fn() == nullptr) return false;
    return true;
}

size_t chunked_workspace_bytes(const ssd_scan_params &p) {
    return ((size_t)p.num_seqs * sizeof(int32_t) + 255) & ~(size_t)255;
}

cudaError_t launch_chunked(const ScanArgs &a, int state_dtype, void *workspace, cudaStream_t stream) {
    switch (state_dtype) {
        case SSD_F32: return launch_typed<float>(a, 0, workspace, stream);
        case SSD_BF16: return launch_typed<__nv_bfloat16>(a, 1, workspace, stream);
        case SSD_F16: return launch_typed<__half>(a, 2, workspace, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssd
