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
// Launch 1 (prep, skipped for unsegmented batches of <= 32 sequences, which the
//   scan kernel sorts itself): sort the sequences by block count, longest
//   first, into the workspace, so the persistent CTAs below take the long
//   chains first; when a batch has few items per SM, also plan the cut of
//   each item into segments run by different CTAs.
// Launch 2 (scan): one persistent CTA per SM.  A work item is one sequence (or
//   one segment of it) and two heads of the same B/C group; its tokens are
//   walked in 128-token blocks.  A segment's initial state is the fp32 state
//   the previous segment's CTA hands over through the workspace.
//   The recurrent state h [2 heads x 64 x 128] never leaves the SM: it lives in
//   tensor memory as an fp32 MMA accumulator.  Per block, with
//   cum_t = sum_{r<=t} dt'_r A (within the block) and Xw_s = exp(cum_end - cum_s) dt'_s x_s:
//     G   = C B^T                          tcgen05, fp32 in TMEM
//     S_h = G o exp(cum_t - cum_s) dt'_s   (s <= t) bf16, written back in TMEM
//     Y   = C h^T                          tcgen05, state entering the block as two
//                                          bf16 parts hi + lo (h - hi), so the fp32
//                                          state enters y at fp32-like accuracy
//     Y  *= exp(cum_t)                     per row and head, in TMEM
//     Y  += S_h X_h                        tcgen05, A operand from TMEM
//     y   = Y + D x                        bf16
//     h   = exp(cum_end) h + B^T Xw        tcgen05 accumulating into the state,
//                                          Xw split into bf16 hi + lo
//   The hi/lo splits keep the state contributions and the state's part of y
//   accurate to ~2^-16, so final states meet fp32-storage accuracy and an fp32
//   initial state reaches y without a bf16 rounding; the intra-block y path
//   runs on bf16 operands with fp32 accumulation.  The state is accumulated in a scaled form with a
//   running per-head scale, so a block needs no rescaling pass over it.  Y is
//   double buffered in TMEM so block k+1's C h^T can start while block k's
//   epilogue drains.
//
// Warp roles (16 warps): warp 0 TMA producer (C, B, X tiles of 128 tokens,
// 4-slot ring); warp 1 issues the output-path MMAs (G, C h^T, S X); warp 2
// owns the TMEM allocation and computes dt softplus, the within-block cumsum
// and the state scales two blocks ahead; warps 4-7 (lane = token) build the
// scaled Xw and issue the state MMAs (B^T Xw); warps 8-11 (lane = token) build
// S and scale the rows of Y; warps 12-15 own the state (lane = state column n:
// bf16 hi/lo copies for C h^T, cache I/O) and write y of the previous block; warp 3
// looks the CTA's items up ahead of use and hands them to the other roles
// through a ring in shared memory.  Hand-offs are mbarriers (and one named
// barrier inside warps 4-7; release/acquire flags in global memory between
// segments);
// every wait is bounded and sets an abort flag plus SSD_DEV_TIMEOUT in
// device_status instead of hanging.
//
// The hot loops are compact (little unrolling): with sixteen warps in six roles
// the kernel's instruction footprint, not its arithmetic, set the block time
// when the loops were unrolled.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstddef>
#include <mutex>
#include <type_traits>

#include "sm100.cuh"
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kQ = 128;            // tokens per block
constexpr int kP = 64;             // head dim
constexpr int kN = 128;            // state dim
constexpr int kSlots = 4;          // TMA ring of 32 KB tiles (C, B, X per block)
constexpr int kTileBytes = 32768;
constexpr int kHalfBytes = 16384;
constexpr int kHbufHead = 8192;    // one head of the half-n bf16 state copy: 64 rows x 128 B
constexpr int kThreads = 512;     // 16 warps, each with exactly one role below
constexpr uint32_t kArrBufs = 3;   // per-block decay arrays in flight (prepared two blocks ahead)

constexpr uint64_t kSpinLimit = 4000000000ull;   // clock cycles (~2 s) per wait
constexpr float kDiagFactorLimit = 80.f;         // |decay| of a 32-token block for the
                                                 // factored diagonal path (e^80 < fp32 max)
constexpr float kScaleLimit = 80.f;              // |exponent| bound of the scaled state inputs
// Segments: long items are cut into segments of `seg` blocks dealt to different
// CTAs, the state handed over in fp32 through the workspace (see prep kernel).
constexpr int kMaxLevels = 32;                   // segments per item at most
constexpr int kMetaInts = 64;                    // [0] items, [1] seg, [2] levels, [4 + j] level offsets
constexpr int kSegMinBlocks = 6;                 // blocks per segment at least
constexpr int kSegPerSm = 8;                     // segments per SM aimed at
constexpr int kSegMaxItemsPerSm = 4;             // batches with more items per SM are not cut
constexpr int kSegSlots = 1024;                  // handed-over states the workspace holds at most
constexpr size_t kSegStateBytes = 2 * 64 * 128 * sizeof(float);   // one head pair's fp32 state

// TMEM columns
constexpr uint32_t kColG = 0;      // G / S (in place), lanes = tokens
constexpr uint32_t kColY = 128;    // Y[2] at 128 + 128 b, lanes = tokens, cols = head x p
constexpr uint32_t kColH = 384;    // state, lanes = n, cols = head x p

constexpr uint32_t kIdG = idesc_bf16(128, 128, false, false);    // C . B^T
constexpr uint32_t kIdY = idesc_bf16(128, 128, false, true);     // C . h^T, h MN-major
constexpr uint32_t kIdSX = idesc_bf16(128, 64, false, true);     // S_h . X_h
constexpr uint32_t kIdH = idesc_bf16(128, 128, true, true);      // B^T . Xw

struct Params {
    int64_t T;
    int32_t S, H, G, hpg, num_items, num_slots;
    int32_t dt_softplus, write_final, state_dtype;
    const float *dt, *dt_bias, *A, *D;
    const int32_t *cu_seqlens, *slot_idx, *order;
    const int32_t *meta, *bstart;                 // segmentation (valid when seg_enabled)
    int32_t *seg_flags;                           // per boundary, head pair and state warp: published
    float *seg_state;                             // per boundary and head pair: fp32 h [2][64][128]
    int32_t seg_enabled;
    int32_t sort_in_cta;                          // S <= 32 and no prep launch: the item warp sorts
    const uint8_t *has_init;
    void *state_cache, *out_y;
    const void *x;
    int32_t *device_status;
    // optional parts of a call
    const int32_t *final_slot_idx;                // NULL: final states to slot_idx
    int64_t slot_stride, final_slot_stride;       // elements between entries (>= 1)
    const int32_t *snap_flag;                     // snapshot pass: initial state copied
    const void *snap_states;                      //   to snap_states[s] (cache dtype)
    void *out_chunk_states;                       // per-chunk states (NULL: off)
    const int32_t *cu_chunks;
    int32_t num_chunk_rows, chunk_size;           // chunk_size a multiple of kQ here
    const uint64_t *sr_seed;                      // fp16 cache: stochastic rounding
    // failure-detection test hooks (see ssd_testing_set_hooks)
    uint64_t spin_limit;                          // clock cycles per wait
    int32_t withhold;                             // hand-over never published, -1: none
};

// per-block decay arrays, written by the dt warp two blocks ahead
//
// The state is accumulated in TMEM in a scaled form hs = h exp(-R): a block
// adds B^T (exp(E - cum_s) dt'_s x_s) with E = -R' and R' the scale in force
// for the block, so no per-block rescale of the accumulator is needed.  R'
// keeps the running scale (R' = R_prev, "fast") while every exponent of the
// block stays within +-kScaleLimit; otherwise the accumulator is renormalised
// to exp(dlt) h before the block (R' = -dlt, exponents <= 0).  After the block
// R = R' + dlt, with dlt the block's total decay cum_end.
struct __align__(16) Arrays {
    float cum[2][kQ];      // [head][token] within-block cumsum of dt' A
    float dtp[2][kQ];      // dt'
    float vfac[2][kQ];     // exp(cum at end of s's 32-block - cum_s) dt'_s
    float vdiag[2][kQ];    // exp(cum before s's 32-block - cum_s) dt'_s
    float cumE[2][4];      // cum at the end of each 32-token block
    float E[2];            // exponent base of the scaled Xw for this block
    float eprev[2];        // exp(R_prev): hs before the block -> h
    float edlt[2];         // exp(dlt)
    float eend[2];         // exp(R after the block): hs after the block -> h
    int32_t renorm[2];     // renormalise the accumulator before this block
    int32_t exact[2][4];   // diagonal block needs the per-element path
};

// One work item: a segment of a sequence for a pair of heads of one B/C group.
struct __align__(16) Item {
    int32_t round;                // deal round after this item
    int32_t seq, h0, g, slot, t0, len, bin, bout;
    int32_t flags;                // bit 0: found, 1: initial state, 2: from the workspace,
                                  // 3: final state to the workspace, 4: initial state
                                  // from the snapshot
    int32_t fslot;                // slot the final state goes to
    int32_t seq_t0;               // first token of the sequence (chunk boundaries)
    int32_t crow;                 // first per-chunk state row of the sequence, -1: none
};
constexpr int kItemRing = 8;      // items looked up ahead by the item warp
constexpr int kSortInCta = 32;    // batches of up to this many sequences are sorted in the kernel
constexpr uint32_t kItemTakers = 15;   // walkers per item: 2 single threads + 13 warps

struct __align__(1024) Smem {
    uint8_t slot[kSlots][kTileBytes];     // TMA ring: C / B [n half][s][n], X [head][s][p]
    uint8_t xw[2][kHalfBytes];            // Xw (hi, then lo), [head][s][p], 128-B swizzle
    uint8_t hbuf[2 * kHbufHead];          // bf16 h (hi part), one half of n at a time: [head][n % 64][p]
    uint8_t hlo[2][2 * kHbufHead];        // bf16 h - hi (lo part), all n: [n / 64][head][n % 64][p]
    Arrays arr[kArrBufs];
    uint64_t full[kSlots], empty[kSlots];
    uint64_t arr_ready[kArrBufs], arr_free[kArrBufs];
    uint64_t g_ready, s_ready, xbuf_free;
    uint64_t hs_a, hs_b, hbuf_a_done, hlo_ready, hlo_free, state_ok, state_done;
    uint64_t yinter_ready, y_scaled, y_ready[2], y_free[2], x_epi_done[2];
    uint64_t drain_y, drain_h;
    uint64_t item_full[kItemRing], item_empty[kItemRing];
    Item items[kItemRing];
    int32_t order_small[kSortInCta];      // longest-first order when the item warp sorts
    uint32_t tmem_base;
    int32_t abort_flag;
    uint64_t spin_limit;          // clock cycles a wait may take before it gives up
};

// Vector (8/16-byte) shared-memory accesses rely on these offsets.
static_assert(sizeof(Arrays) % 16 == 0, "Arrays must keep float4 rows aligned");
static_assert(offsetof(Arrays, dtp) % 16 == 0 && offsetof(Arrays, vfac) % 16 == 0 &&
              offsetof(Arrays, vdiag) % 16 == 0, "Arrays rows must be 16-byte aligned");
static_assert(offsetof(Smem, arr) % 16 == 0, "Arrays must start 16-byte aligned");
static_assert(offsetof(Smem, xw) % 1024 == 0 && offsetof(Smem, hbuf) % 1024 == 0 &&
              offsetof(Smem, hlo) % 1024 == 0,
              "swizzled operand tiles must be 1024-byte aligned");

// ---------------------------------------------------------------------------
// work enumeration, identical in every role
// ---------------------------------------------------------------------------
struct Chunk {
    int32_t seq, h0, g, slot, fslot, seq_t0, crow;
    int32_t row0;        // first token of this block (total tokens < 2^31 on this path)
    int32_t l;           // valid tokens in this block
    int32_t bin, bout;   // workspace state slots read at the first / written at the last block
    bool init, first, last, empty_item;
    bool init_ws;        // the initial state comes from the workspace (a previous segment)
    bool fin_ws;         // the final state goes to the workspace (a following segment)
    bool snap;           // the initial state comes from the snapshot of the cache slot
};

// Next valid item of this CTA (longest sequences first, snake order over the
// CTAs), starting at deal round `round`.  With segmentation the items are
// dealt level by level -- every item's first segment, then every second
// segment, ... -- so a segment's predecessor is always dealt earlier; the
// sequences with a j-th segment are a prefix of the longest-first order.
// Out of line: called once per item.
__device__ __noinline__ Item find_item(const Params &p, const int32_t *order, int32_t round, bool report) {
    Item it;
    it.flags = 0;
    const int32_t hp_per_seq = p.H / 2;
    const int32_t grid = gridDim.x, cta = blockIdx.x;
    const int32_t num_items = p.seg_enabled ? p.meta[0] : p.num_items;
    const int32_t seg = p.seg_enabled ? p.meta[1] : 0x40000000;
    const int32_t nlev = p.seg_enabled ? p.meta[2] : 1;
    while (true) {
        const int32_t base = round * grid;
        const int32_t idx = base + ((round & 1) ? (grid - 1 - cta) : cta);
        ++round;
        if (base >= num_items) break;
        if (idx >= num_items) continue;
        int32_t j = 0, off = 0;
        if (p.seg_enabled) {
            while (j + 1 < nlev && idx >= p.meta[4 + j + 1]) ++j;
            off = p.meta[4 + j];
        }
        const int32_t r = idx - off;
        const int32_t rank = r / hp_per_seq;
        const int32_t hp = r - rank * hp_per_seq;
        const int32_t seq = order[rank];
        const int32_t h0 = hp * 2;
        // every per-sequence entry the item may need, loaded together (one
        // memory round trip instead of a chain of dependent ones)
        const int64_t a = p.cu_seqlens[seq], e = p.cu_seqlens[seq + 1];
        const bool init_raw = p.has_init != nullptr && p.has_init[seq] != 0;
        const int32_t slot_raw = p.slot_idx != nullptr ? p.slot_idx[seq * p.slot_stride] : 0;
        const int32_t fslot_raw = p.final_slot_idx != nullptr ? p.final_slot_idx[seq * p.final_slot_stride] : 0;
        const bool snap_raw = p.snap_flag != nullptr && p.snap_flag[seq] != 0;
        const int64_t c0 = p.out_chunk_states ? p.cu_chunks[seq] : 0;
        const int64_t c1 = p.out_chunk_states ? p.cu_chunks[seq + 1] : 0;
        if (a < 0 || e < a || e > p.T) {
            if (report && j == 0 && p.device_status) atomicOr(p.device_status, SSD_DEV_BAD_SEQLENS);
            continue;
        }
        const bool init = init_raw;
        int32_t slot = 0, fslot = 0;
        if (init || p.write_final) {
            slot = slot_raw;
            fslot = (p.write_final && p.final_slot_idx) ? fslot_raw : slot;
            if ((init && (slot < 0 || slot >= p.num_slots)) ||
                (p.write_final && (fslot < 0 || fslot >= p.num_slots))) {
                if (report && j == 0 && p.device_status) atomicOr(p.device_status, SSD_DEV_BAD_SLOT);
                continue;
            }
        }
        const int32_t len = (int32_t)(e - a);
        int32_t crow = -1;
        if (p.out_chunk_states) {
            if (c0 >= 0 && c1 - c0 == (len + p.chunk_size - 1) / p.chunk_size && c1 <= p.num_chunk_rows)
                crow = (int32_t)c0;
            else if (report && j == 0 && p.device_status)
                atomicOr(p.device_status, SSD_DEV_BAD_CHUNKS);
        }
        const bool snap = init && snap_raw;
        const int32_t nb = (len + kQ - 1) / kQ;
        const int32_t nseg = nb == 0 ? 1 : (nb + seg - 1) / seg;
        const int32_t b0 = j * seg, b1 = min(nb, (j + 1) * seg);
        it.seq = seq;
        it.h0 = h0;
        it.g = h0 / p.hpg;
        it.slot = slot;
        it.t0 = (int32_t)a + b0 * kQ;
        it.len = nb == 0 ? 0 : min(len, b1 * kQ) - b0 * kQ;
        it.bin = j > 0 ? (p.bstart[rank] + j - 1) * hp_per_seq + hp : 0;
        it.bout = j + 1 < nseg ? (p.bstart[rank] + j) * hp_per_seq + hp : 0;
        it.flags = 1 | ((j > 0 || init) ? 2 : 0) | (j > 0 ? 4 : 0) | (j + 1 < nseg ? 8 : 0) |
                   ((j == 0 && snap) ? 16 : 0);
        it.fslot = fslot;
        it.seq_t0 = (int32_t)a;
        it.crow = crow;
        break;
    }
    it.round = round;
    return it;
}


// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
// The waits test the barrier once inline; the bounded spin is out of line so
// that the many call sites stay small (the whole kernel's hot code has to fit
// the SM's instruction cache).
__device__ __noinline__ bool wait_bar_slow(Smem &sm, uint64_t *bar, uint32_t parity, int32_t *status) {
    const uint64_t t_start = clock64();
    uint32_t it = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++it & 255u) == 0) {
            if (*(volatile int32_t *)&sm.abort_flag) return false;
            if (clock64() - t_start > sm.spin_limit) {
                atomicExch(&sm.abort_flag, 1);
                if (status) atomicOr(status, SSD_DEV_TIMEOUT);
                return false;
            }
        }
    }
    return true;
}

// Wait for this CTA's own asynchronous work (TMA loads, MMAs) before it exits.
// Bounded like every wait, but not cut short by the abort flag: that work ends
// by itself and must not outlive the CTA's shared and tensor memory.
__device__ __noinline__ void drain_wait(uint64_t *bar, uint32_t parity, int32_t *status) {
    const uint64_t t_start = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t_start > kSpinLimit) {
            if (status) atomicOr(status, SSD_DEV_TIMEOUT);
            return;
        }
    }
}

// Single-thread wait (producer / MMA issuer).
__device__ __forceinline__ bool wait_bar(Smem &sm, uint64_t *bar, uint32_t parity, int32_t *status) {
    return mbar_try_wait(bar, parity) || wait_bar_slow(sm, bar, parity, status);
}

__device__ __noinline__ bool warp_wait_slow(Smem &sm, uint64_t *bar, uint32_t parity, int32_t *status) {
    const uint64_t t_start = clock64();
    uint32_t it = 0;
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if ((++it & 255u) == 0) {
            int give_up = 0;
            if ((threadIdx.x & 31) == 0) {
                if (*(volatile int32_t *)&sm.abort_flag) {
                    give_up = 1;
                } else if (clock64() - t_start > sm.spin_limit) {
                    atomicExch(&sm.abort_flag, 1);
                    if (status) atomicOr(status, SSD_DEV_TIMEOUT);
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
    }
}

// Whole-warp wait with a warp-uniform result (all 32 lanes must call it).
// A barrier phase never runs two completions ahead of its slowest waiter in
// this kernel, so once one lane observes completion every lane will.
__device__ __forceinline__ bool warp_wait(Smem &sm, uint64_t *bar, uint32_t parity, int32_t *status) {
    return __all_sync(0xffffffffu, mbar_try_wait(bar, parity)) || warp_wait_slow(sm, bar, parity, status);
}

__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t *f) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int32_t *f, int32_t v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

// Whole-warp wait until another CTA has published a segment's final state
// (every lane acquires the flag itself).  Bounded like the barrier waits.
__device__ __noinline__ bool warp_wait_flag(Smem &sm, const int32_t *flag, int32_t *status) {
    const uint64_t t_start = clock64();
    uint32_t it = 0;
    while (!__all_sync(0xffffffffu, ld_acquire_gpu(flag) != 0)) {
        if ((++it & 63u) == 0) {
            int give_up = 0;
            if ((threadIdx.x & 31) == 0) {
                if (*(volatile int32_t *)&sm.abort_flag) {
                    give_up = 1;
                } else if (clock64() - t_start > sm.spin_limit) {
                    atomicExch(&sm.abort_flag, 1);
                    if (status) atomicOr(status, SSD_DEV_TIMEOUT);
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
        __nanosleep(32);
    }
    return true;
}

// The ik-th item of this CTA from the ring (flags 0: no more items, or the
// wait gave up).  Out of line: called once per item in every role.
__device__ __noinline__ Item take_item(Smem &sm, uint32_t ik, bool whole_warp, int32_t *status) {
    const uint32_t s = ik % kItemRing, par = (ik / kItemRing) & 1;
    Item it;
    if (!(whole_warp ? warp_wait(sm, &sm.item_full[s], par, status)
                     : wait_bar(sm, &sm.item_full[s], par, status))) {
        it.flags = 0;
        return it;
    }
    it = sm.items[s];
    if (whole_warp) __syncwarp();
    if (!whole_warp || (threadIdx.x & 31) == 0) mbar_arrive(&sm.item_empty[s]);
    return it;
}

// Longest-first order of a batch of at most 32 sequences by a bitonic sort
// over the lanes of one warp (keys as in the prep kernel).  Out of line and
// compact: runs once per CTA.
__device__ __noinline__ void sort_small(const Params &p, int32_t *order) {
    const int lane = threadIdx.x & 31;
    unsigned long long key = ~0ull;
    if (lane < p.S) {
        const int64_t a = p.cu_seqlens[lane], e = p.cu_seqlens[lane + 1];
        const int32_t v = (a < 0 || e < a || e > p.T) ? 0 : (int32_t)((e - a + kQ - 1) / kQ);
        key = ((unsigned long long)(uint32_t)(0x7FFFFFFF - v) << 32) | (uint32_t)lane;
    }
#pragma unroll 1
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll 1
        for (int j = k >> 1; j > 0; j >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, j);
            key = (((lane & j) == 0) == ((lane & k) == 0)) ? (o < key ? o : key) : (o > key ? o : key);
        }
    }
    order[lane] = (int32_t)(uint32_t)key;
    __syncwarp();
}

// Walks this CTA's items block by block; identical in every role.  The items
// come from a ring in shared memory that the item warp fills ahead of use,
// so no role waits on the lookups' global loads at an item boundary.
// whole_warp: all 32 lanes of a warp walk together (else one thread alone).
struct Walker {
    Item it;
    int32_t nb = 0, b = 0;
    uint32_t ik = 0;              // items taken from the ring
    bool have = false;

    __device__ void fill(Chunk &c) const {
        c.seq = it.seq; c.h0 = it.h0; c.g = it.g; c.slot = it.slot;
        c.fslot = it.fslot; c.seq_t0 = it.seq_t0; c.crow = it.crow;
        c.init = (it.flags & 2) != 0;
        c.init_ws = (it.flags & 4) != 0;
        c.fin_ws = (it.flags & 8) != 0;
        c.snap = (it.flags & 16) != 0;
        c.bin = it.bin;
        c.bout = it.bout;
    }

    __device__ bool take(Smem &sm, bool whole_warp, int32_t *status) {
        it = take_item(sm, ik++, whole_warp, status);
        return (it.flags & 1) != 0;
    }

    // Next event: a block of an item, or (if want_empty) an item without tokens.
    __device__ bool next(Smem &sm, Chunk &c, bool want_empty, bool whole_warp, int32_t *status) {
        while (true) {
            if (!have || b >= nb) {
                if (!take(sm, whole_warp, status)) return false;
                have = true;
                nb = (it.len + kQ - 1) / kQ;
                b = 0;
                if (nb == 0) {
                    if (want_empty) {
                        fill(c);
                        c.row0 = it.t0; c.l = 0;
                        c.first = c.last = true; c.empty_item = true;
                        return true;
                    }
                    continue;
                }
            }
            fill(c);
            c.row0 = it.t0 + b * kQ;
            c.l = min(kQ, it.len - b * kQ);
            c.first = (b == 0);
            c.last = (b == nb - 1);
            c.empty_item = false;
            ++b;
            return true;
        }
    }
};

// Barrier over the four Xw warps (named barrier 1) that also ANDs a flag over
// them, so that the group takes every exit together.
__device__ __forceinline__ bool xw_group_and(bool v) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)v) : "memory");
    return r != 0;
}

__device__ __noinline__ float softplus_f(float z) {
    return fmaxf(z, 0.f) + log1pf(__expf(-fabsf(z)));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename StT> __device__ __forceinline__ float load_state(const StT *p);
template <> __device__ __forceinline__ float load_state<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float load_state<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
template <> __device__ __forceinline__ float load_state<__half>(const __half *p) {
    return __half2float(*p);
}
template <typename StT> __device__ __forceinline__ void store_state(StT *p, float v);
template <> __device__ __forceinline__ void store_state<float>(float *p, float v) { *p = v; }
template <> __device__ __forceinline__ void store_state<__nv_bfloat16>(__nv_bfloat16 *p, float v) {
    *p = __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ void store_state<__half>(__half *p, float v) {
    *p = __float2half_rn(v);
}
// One state value at flat element index e of a [rows, H, P, N] tensor: nearest
// even, or for fp16 with a seed stochastic rounding with the element's Philox
// word (stream 0: the cache, 1: per-chunk states).
// Out of line: the generator's ten rounds stay out of the state warps' hot code.
__device__ __noinline__ void put_state_sr(__half *base, int64_t e, float v, uint64_t seed, uint32_t stream) {
    base[e] = sr_f16(v, sr_word(sr_block(seed, (uint64_t)e >> 2, stream), (uint32_t)(e & 3)));
}
template <typename StT>
__device__ __forceinline__ void put_state(StT *base, int64_t e, float v, bool sr, uint64_t seed, uint32_t stream) {
    if constexpr (std::is_same<StT, __half>::value) {
        if (sr) {
            put_state_sr(base, e, v, seed, stream);
            return;
        }
    }
    store_state<StT>(base + e, v);
}

// ---------------------------------------------------------------------------
// launch 1: longest-first order of the sequences
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 1024;
constexpr int kSortMax = 8192;
constexpr int kPrepSmem = kSortMax * (int)sizeof(unsigned long long);   // dynamic shared memory of the prep kernel

// Longest-first order of the sequences (by block count), and, when enabled,
// their cut into segments: seg blocks per segment, chosen so that about
// kSegPerSm segments fall to each SM when the longest item is shorter than an
// SM's mean share of the blocks (long equal items otherwise leave most SMs idle
// in the last deal round); at most kMaxLevels segments per item, at least
// kSegMinBlocks blocks per segment and at most `cap` handed-over states
// (boundaries x head pairs, the workspace's capacity).  Writes order[S], and
// with segmentation meta
// (item count, seg, levels, level offsets), bstart[rank] (first boundary of
// each sequence) and clears the boundary flags of this call.  Run by CTA 0.
__device__ __noinline__ void prep_order(const int32_t *cu, int S, int64_t T, int32_t *order, int32_t *meta,
                                        int32_t *bstart, int32_t *flags, int hp, int num_sms, int cap,
                                        int seg_enabled) {
    // sort keys: (2^31 - 1 - block count) << 32 | sequence, ascending = longest
    // first, ties by sequence index
    extern __shared__ unsigned long long keys[];
    auto nbr = [&](int r) { return 0x7FFFFFFF - (int32_t)(keys[r] >> 32); };   // block count by rank
    __shared__ int32_t part[kPrepThreads / 32];
    __shared__ uint32_t total;                   // blocks of all sequences (< 2^25 here)
    __shared__ int32_t seg_s;
    if (S > kSortMax) {
        for (int s = threadIdx.x; s < S; s += blockDim.x) order[s] = s;
        return;
    }
    int p2 = 1;                                  // bitonic sort over a power of two
    while (p2 < S) p2 <<= 1;
    for (int s = threadIdx.x; s < p2; s += blockDim.x) {
        unsigned long long key = ~0ull;          // padding sorts last
        if (s < S) {
            const int64_t a = cu[s], e = cu[s + 1];
            const int32_t v = (a < 0 || e < a || e > T) ? 0 : (int32_t)((e - a + kQ - 1) / kQ);
            key = ((unsigned long long)(uint32_t)(0x7FFFFFFF - v) << 32) | (uint32_t)s;
        }
        keys[s] = key;
    }
    if (threadIdx.x == 0) total = 0;
    __syncthreads();
    for (int k = 2; k <= p2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < p2; i += blockDim.x) {
                const int l = i ^ j;
                if (l > i) {
                    const unsigned long long x = keys[i], y = keys[l];
                    if ((x > y) == ((i & k) == 0)) {
                        keys[i] = y;
                        keys[l] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
    uint32_t mine = 0;
    for (int r = threadIdx.x; r < S; r += blockDim.x) {
        order[r] = (int32_t)(uint32_t)keys[r];
        mine += nbr(r);
    }
    if (!seg_enabled) return;
    mine = __reduce_add_sync(0xffffffffu, mine);
    if ((threadIdx.x & 31) == 0 && mine) atomicAdd(&total, mine);
    __syncthreads();
    if (threadIdx.x == 0) {
        const long long work = (long long)total * hp;
        int seg = 0x40000000;
        // Only when the longest item is shorter than an SM's mean share: a
        // longer one is the critical path already, and its segments would run
        // one after another anyway.
        if (cap > 0 && (long long)nbr(0) * num_sms < work) {
            // boundaries x hp <= total x hp / seg <= cap
            long long v = max((long long)kSegMinBlocks, (work + (long long)kSegPerSm * num_sms - 1) / ((long long)kSegPerSm * num_sms));
            v = max(v, (work + cap - 1) / cap);
            v = max(v, (long long)(nbr(0) + kMaxLevels - 1) / kMaxLevels);
            seg = (int)min(v, 0x40000000LL);
        }
        seg_s = seg;
    }
    __syncthreads();
    const int seg = seg_s;
    // boundaries per rank: nseg - 1; exclusive prefix sum into bstart
    constexpr int kPer = kSortMax / kPrepThreads;
    const int r0 = threadIdx.x * kPer;
    int32_t local = 0;
    for (int k = 0; k < kPer; ++k) {
        const int r = r0 + k;
        if (r < S) local += nbr(r) == 0 ? 0 : (nbr(r) + seg - 1) / seg - 1;
    }
    // block-wide exclusive scan of `local`
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int32_t incl = local;
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) part[w] = incl;
    __syncthreads();
    if (w == 0) {
        int32_t v = part[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        part[lane] = v;                          // inclusive over warps
    }
    __syncthreads();
    int32_t run = (w ? part[w - 1] : 0) + incl - local;
    for (int k = 0; k < kPer; ++k) {
        const int r = r0 + k;
        if (r < S) {
            bstart[r] = run;
            run += nbr(r) == 0 ? 0 : (nbr(r) + seg - 1) / seg - 1;
        }
    }
    const int32_t nbound = part[31];
    for (int i = threadIdx.x; i < nbound * hp * 4; i += blockDim.x) flags[i] = 0;
    if (threadIdx.x == 0) {
        const int nlev = nbr(0) == 0 ? 1 : (nbr(0) + seg - 1) / seg;
        // sequences with a j-th segment are the first cnt_j ranks (block counts are sorted)
        int32_t offs = 0;
        for (int j = 0; j < nlev; ++j) {
            meta[4 + j] = offs;
            int lo = 0, hi = S;                  // first rank whose item has no j-th segment
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                const int ns = nbr(mid) == 0 ? 1 : (nbr(mid) + seg - 1) / seg;
                if (ns > j) lo = mid + 1; else hi = mid;
            }
            offs += lo * hp;
        }
        meta[4 + nlev] = offs;
        meta[0] = offs;
        meta[1] = seg;
        meta[2] = nlev;
    }
}

// Launch 1: the order (CTA 0, when the scan kernel does not sort the batch
// itself) and, for calls whose sequences may read a slot another sequence
// writes, the snapshot of those initial states (every CTA, a sequence each).
__global__ void __launch_bounds__(kPrepThreads) prep_order_kernel(const int32_t *cu, int S, int64_t T,
                                                                    int32_t *order, int32_t *meta,
                                                                    int32_t *bstart, int32_t *flags, int hp,
                                                                    int num_sms, int cap, int seg_enabled,
                                                                    int do_sort, SnapshotArgs snap,
                                                                    int do_snap) {
    if (do_sort && blockIdx.x == 0) prep_order(cu, S, T, order, meta, bstart, flags, hp, num_sms, cap, seg_enabled);
    if (do_snap) {
        __shared__ int conflict;
        for (int s = blockIdx.x; s < snap.S; s += gridDim.x) snapshot_sequence(snap, s, &conflict);
    }
}

// ---------------------------------------------------------------------------
// launch 2: the scan
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 f2(uint32_t a, uint32_t b) {
    return make_float2(__uint_as_float(a), __uint_as_float(b));
}
__device__ __forceinline__ uint32_t pack2(float2 v) { return pack_bf16(v.x, v.y); }

// S on the diagonal 32-token block when its decay is too steep for the
// factored form: exp(cum_t - cum_s) dt'_s per element, for the 16 tokens s of
// half-block c16; G is read from, and S_h written back to, the 16 TMEM columns
// at taddr (head h at +8h).  Rare; out of line.
__device__ __noinline__ void s_diag_exact(uint32_t taddr, const Arrays &ar, int t, int c16, float cum_t0,
                                          float cum_t1) {
    uint32_t g[16], out0[8], out1[8];
    tmem_ld16(taddr, g);
    tmem_wait_ld();
#pragma unroll
    for (int i2 = 0; i2 < 8; ++i2) {
        const int s = 16 * c16 + 2 * i2;
        float r0[2], r1[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float gv = __uint_as_float(g[2 * i2 + e]);
            const bool keep = (s + e) <= t;
            r0[e] = keep ? gv * (__expf(cum_t0 - ar.cum[0][s + e]) * ar.dtp[0][s + e]) : 0.f;
            r1[e] = keep ? gv * (__expf(cum_t1 - ar.cum[1][s + e]) * ar.dtp[1][s + e]) : 0.f;
        }
        out0[i2] = pack_bf16(r0[0], r0[1]);
        out1[i2] = pack_bf16(r1[0], r1[1]);
    }
    tmem_st8(taddr, out0);
    tmem_st8(taddr + 8, out1);
}

// dt softplus, the within-block cumsum of dt' A and the per-block scales of one
// block, computed by one warp into sm.arr[k % kArrBufs]: four passes over the
// 32-token sub-blocks, one token per lane, the cumsum carried across passes.
// The block's dt values come in `dr`, loaded a block earlier by the caller.
// R0/R1 carry the running scale of the state accumulator per head (0 at the
// first block of an item).
struct DtOut {
    float R0, R1;
    int32_t ok;
};
// dt of tokens 32 jb + lane (jb = 0..3) of a block, heads h0 and h0 + 1.
struct DtRaw {
    float2 v0, v1, v2, v3;
};
__device__ __forceinline__ DtRaw dt_load(const Params &p, int32_t row0, int32_t l, int32_t h0) {
    const int lane = threadIdx.x & 31;
    auto ld = [&](int jb) {
        const int tok = 32 * jb + lane;
        return tok < l ? __ldg(reinterpret_cast<const float2 *>(p.dt + (int64_t)(row0 + tok) * p.H + h0))
                       : make_float2(0.f, 0.f);
    };
    DtRaw d;
    d.v0 = ld(0);
    d.v1 = ld(1);
    d.v2 = ld(2);
    d.v3 = ld(3);
    return d;
}
__device__ __forceinline__ DtOut dt_prep(Smem &sm, const Params &p, const DtRaw &dr, int32_t l, int32_t h0,
                                         bool first, uint32_t k, float R0, float R1, int32_t *status) {
    const int lane = threadIdx.x & 31;
    DtOut out;
    out.R0 = first ? 0.f : R0;
    out.R1 = first ? 0.f : R1;
    out.ok = 0;
    const uint32_t ab = k % kArrBufs, use = k / kArrBufs;
    Arrays &ar = sm.arr[ab];
    const float bias0 = p.dt_bias ? p.dt_bias[h0] : 0.f, bias1 = p.dt_bias ? p.dt_bias[h0 + 1] : 0.f;
    const float A0 = p.A[h0], A1 = p.A[h0 + 1];
    if (use > 0 && !warp_wait(sm, &sm.arr_free[ab], (use - 1) & 1, status)) return out;
    float carry0 = 0.f, carry1 = 0.f;             // cum at the end of the previous sub-block
    float lo0 = 0.f, hi0 = 0.f, lo1 = 0.f, hi1 = 0.f;
#pragma unroll 1
    for (int jb = 0; jb < 4; ++jb) {
        const int tok = 32 * jb + lane;
        const bool valid = tok < l;
        const float2 raw = jb == 0 ? dr.v0 : jb == 1 ? dr.v1 : jb == 2 ? dr.v2 : dr.v3;
        const float z0 = raw.x + bias0, z1 = raw.y + bias1;
        const float d0 = valid ? (p.dt_softplus ? softplus_f(z0) : z0) : 0.f;
        const float d1 = valid ? (p.dt_softplus ? softplus_f(z1) : z1) : 0.f;
        float s0 = d0 * A0, s1 = d1 * A1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float v0 = __shfl_up_sync(0xffffffffu, s0, off);
            const float v1 = __shfl_up_sync(0xffffffffu, s1, off);
            if (lane >= off) { s0 += v0; s1 += v1; }
        }
        const float c0 = carry0 + s0, c1 = carry1 + s1;
        const float end0 = __shfl_sync(0xffffffffu, c0, 31), end1 = __shfl_sync(0xffffffffu, c1, 31);
        ar.cum[0][tok] = c0;
        ar.cum[1][tok] = c1;
        ar.dtp[0][tok] = d0;
        ar.dtp[1][tok] = d1;
        ar.vfac[0][tok] = d0 != 0.f ? __expf(end0 - c0) * d0 : 0.f;
        ar.vfac[1][tok] = d1 != 0.f ? __expf(end1 - c1) * d1 : 0.f;
        ar.vdiag[0][tok] = d0 != 0.f ? __expf(fminf(carry0 - c0, kDiagFactorLimit)) * d0 : 0.f;
        ar.vdiag[1][tok] = d1 != 0.f ? __expf(fminf(carry1 - c1, kDiagFactorLimit)) * d1 : 0.f;
        lo0 = fminf(lo0, c0); hi0 = fmaxf(hi0, c0);
        lo1 = fminf(lo1, c1); hi1 = fmaxf(hi1, c1);
        if (lane == 0) {
            ar.cumE[0][jb] = end0;
            ar.cumE[1][jb] = end1;
            ar.exact[0][jb] = fabsf(end0 - carry0) > kDiagFactorLimit;
            ar.exact[1][jb] = fabsf(end1 - carry1) > kDiagFactorLimit;
        }
        carry0 = end0;
        carry1 = end1;
    }
    // block extremes of cum (the exponent range of the scaled state inputs)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        lo0 = fminf(lo0, __shfl_xor_sync(0xffffffffu, lo0, off));
        hi0 = fmaxf(hi0, __shfl_xor_sync(0xffffffffu, hi0, off));
        lo1 = fminf(lo1, __shfl_xor_sync(0xffffffffu, lo1, off));
        hi1 = fmaxf(hi1, __shfl_xor_sync(0xffffffffu, hi1, off));
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        float &R = hh ? out.R1 : out.R0;
        const float dlt = hh ? carry1 : carry0;
        const float lo = hh ? lo1 : lo0, hi = hh ? hi1 : hi0;
        const bool fast = (-R - lo <= kScaleLimit) && (-R - hi >= -kScaleLimit);
        const float Rp = fast ? R : -dlt;          // scale in force for this block
        if (lane == 0) {
            ar.E[hh] = -Rp;
            ar.eprev[hh] = __expf(R);
            ar.edlt[hh] = __expf(dlt);
            ar.eend[hh] = __expf(Rp + dlt);
            ar.renorm[hh] = fast ? 0 : 1;
        }
        R = Rp + dlt;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.arr_ready[ab]);
    out.ok = 1;
    return out;
}

template <typename StT>
__global__ void __launch_bounds__(kThreads, 1)
chunked_scan_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ CUtensorMap map_c, const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) { mbar_init(&sm.full[i], 1); mbar_init(&sm.empty[i], 2); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.y_free[i], 4);
            mbar_init(&sm.y_ready[i], 1);
            mbar_init(&sm.x_epi_done[i], 4);
        }
        for (uint32_t i = 0; i < kArrBufs; ++i) {
            mbar_init(&sm.arr_ready[i], 1);
            mbar_init(&sm.arr_free[i], 12);
        }
        mbar_init(&sm.g_ready, 1);
        mbar_init(&sm.s_ready, 4);
        mbar_init(&sm.xbuf_free, 1);
        mbar_init(&sm.hs_a, 2);
        mbar_init(&sm.hs_b, 2);
        mbar_init(&sm.hbuf_a_done, 1);
        mbar_init(&sm.hlo_ready, 4);
        mbar_init(&sm.hlo_free, 1);
        mbar_init(&sm.state_ok, 4);
        mbar_init(&sm.state_done, 1);
        mbar_init(&sm.yinter_ready, 1);
        mbar_init(&sm.y_scaled, 4);
        mbar_init(&sm.drain_y, 1);
        mbar_init(&sm.drain_h, 1);
        for (int i = 0; i < kItemRing; ++i) {
            mbar_init(&sm.item_full[i], 1);
            mbar_init(&sm.item_empty[i], kItemTakers);
        }
        sm.abort_flag = 0;
        sm.spin_limit = p.spin_limit;
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

    if (warp < 4) {
      if (warp == 0) {
        // ===================== TMA producer =====================
        if (lane == 0) {
            tma_prefetch_desc(&map_x);
            tma_prefetch_desc(&map_b);
            tma_prefetch_desc(&map_c);
            Walker wk;
            Chunk c;
            uint32_t kc = 0, issued = 0;
            bool ok = true;
            while (ok && wk.next(sm, c, false, false, status)) {
                const int32_t row = c.row0;
#pragma unroll 1
                for (int j = 0; j < 3; ++j) {                    // C, B, X
                    const uint32_t tile = 3 * kc + j, slot = tile % kSlots, use = tile / kSlots;
                    const CUtensorMap *m = (j == 0) ? &map_c : (j == 1) ? &map_b : &map_x;
                    const int32_t c0 = (j == 2) ? c.h0 * kP : c.g * kN;
                    const int32_t c1 = (j == 2) ? (c.h0 + 1) * kP : c.g * kN + 64;
                    if (use > 0 && !mbar_try_wait(&sm.empty[slot], (use - 1) & 1)) {
                        // slot still busy: warm L2 with this tile while waiting
                        tma_prefetch_l2_2d(m, c0, row);
                        tma_prefetch_l2_2d(m, c1, row);
                        if (!(ok = wait_bar(sm, &sm.empty[slot], (use - 1) & 1, status))) break;
                    }
                    if (use > 0 && (tile - kSlots) % 3 == 2) {
                        // previous occupant was an X tile: the epilogue also reads it
                        const uint32_t pk = (tile - kSlots) / 3;
                        if (!(ok = wait_bar(sm, &sm.x_epi_done[pk & 1], (pk >> 1) & 1, status))) break;
                    }
                    mbar_arrive_expect_tx(&sm.full[slot], kTileBytes);
                    uint8_t *dst = sm.slot[slot];
                    tma_load_2d(dst, m, &sm.full[slot], c0, row);
                    tma_load_2d(dst + kHalfBytes, m, &sm.full[slot], c1, row);
                    issued = tile + 1;
                }
                ++kc;
            }
            for (uint32_t t = (issued > (uint32_t)kSlots ? issued - kSlots : 0); t < issued; ++t)
                drain_wait(&sm.full[t % kSlots], (t / kSlots) & 1, status);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer, output path =====================
        if (lane == 0) {
            Walker wk;
            Chunk c;
            uint32_t kc = 0;
            bool ok = true;
            const uint32_t bH = smem_u32(sm.hbuf);
            while (ok && wk.next(sm, c, false, false, status)) {
                const uint32_t tC = 3 * kc, tB = 3 * kc + 1, tX = 3 * kc + 2;
                const uint32_t bC = smem_u32(sm.slot[tC % kSlots]);
                const uint32_t bB = smem_u32(sm.slot[tB % kSlots]);
                const uint32_t bX = smem_u32(sm.slot[tX % kSlots]);
                const uint32_t ycol = kColY + 128 * (kc & 1);
                // ---- G = C B^T ----
                if (!(ok = wait_bar(sm, &sm.full[tC % kSlots], (tC / kSlots) & 1, status) &&
                           wait_bar(sm, &sm.full[tB % kSlots], (tB / kSlots) & 1, status)))
                    break;
                tc_fence_after();
                {
                    const uint64_t dc = smem_desc_sw128(bC, 16, 1024), db = smem_desc_sw128(bB, 16, 1024);
#pragma unroll
                    for (uint32_t ks = 0; ks < 8; ++ks) {
                        const uint32_t off = ((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
                        mma_ss(tmem + kColG, dc + off, db + off, kIdG, ks > 0);
                    }
                }
                mma_commit(&sm.g_ready);
                mma_commit(&sm.empty[tB % kSlots]);              // this path's only read of B
                // ---- Y[b] = C h^T, first half of the state columns n ----
                if (!(ok = wait_bar(sm, &sm.hs_a, kc & 1, status) &&
                           (kc < 2 || wait_bar(sm, &sm.y_free[kc & 1], ((kc >> 1) - 1) & 1, status))))
                    break;
                tc_fence_after();
                {
                    const uint64_t dc = smem_desc_sw128(bC, 16, 1024), dh = smem_desc_sw128(bH, kHbufHead, 1024);
#pragma unroll
                    for (uint32_t ks = 0; ks < 4; ++ks)
                        mma_ss(tmem + ycol, dc + ks * 2, dh + ks * 128, kIdY, ks > 0);
                }
                mma_commit(&sm.hbuf_a_done);
                // ---- Y[b] += C h^T, second half of n ----
                if (!(ok = wait_bar(sm, &sm.hs_b, kc & 1, status))) break;
                tc_fence_after();
                {
                    const uint64_t dc = smem_desc_sw128(bC + kHalfBytes, 16, 1024), dh = smem_desc_sw128(bH, kHbufHead, 1024);
#pragma unroll
                    for (uint32_t ks = 0; ks < 4; ++ks)
                        mma_ss(tmem + ycol, dc + ks * 2, dh + ks * 128, kIdY, 1);
                }
                // ---- Y[b] += C h_lo^T: the low bf16 part of the fp32 state, all n ----
                if (!(ok = wait_bar(sm, &sm.hlo_ready, kc & 1, status))) break;
                tc_fence_after();
#pragma unroll
                for (uint32_t j = 0; j < 2; ++j) {
                    const uint64_t dc = smem_desc_sw128(bC + j * kHalfBytes, 16, 1024);
                    const uint64_t dh = smem_desc_sw128(smem_u32(sm.hlo[j]), kHbufHead, 1024);
#pragma unroll
                    for (uint32_t ks = 0; ks < 4; ++ks)
                        mma_ss(tmem + ycol, dc + ks * 2, dh + ks * 128, kIdY, 1);
                }
                mma_commit(&sm.yinter_ready);
                mma_commit(&sm.hlo_free);
                mma_commit(&sm.empty[tC % kSlots]);
                mma_commit(&sm.empty[tC % kSlots]);
                // ---- Y[b] += S_h X_h ----
                if (!(ok = wait_bar(sm, &sm.full[tX % kSlots], (tX / kSlots) & 1, status) &&
                           wait_bar(sm, &sm.s_ready, kc & 1, status) &&
                           wait_bar(sm, &sm.y_scaled, kc & 1, status)))
                    break;
                tc_fence_after();
                {
                    const uint64_t dx = smem_desc_sw128(bX, 1024, 1024);
#pragma unroll
                    for (uint32_t i = 0; i < 16; ++i) {
                        const uint32_t hh = i >> 3, ks = i & 7;
                        const uint32_t acol = kColG + 16 * ks + 8 * hh;     // S_h, tokens 16ks..16ks+15
                        mma_ts(tmem + ycol + 64 * hh, tmem + acol, dx + ((hh * kHalfBytes + ks * 2048) >> 4), kIdSX, 1);
                    }
                }
                mma_commit(&sm.y_ready[kc & 1]);
                mma_commit(&sm.empty[tX % kSlots]);
                ++kc;
            }
            mma_commit(&sm.drain_y);
            drain_wait(&sm.drain_y, 0, status);
        }
    } else if (warp == 3) {
        // ===================== item dealer =====================
        // Looks this CTA's items up in deal order (one thread) and hands them to
        // the walkers of every role through the ring, up to kItemRing ahead;
        // the last entry is the end marker.
        const int32_t *order = p.order;
        if (p.sort_in_cta) {
            sort_small(p, sm.order_small);
            order = sm.order_small;
        }
        if (lane == 0) {
            int32_t round = 0;
            for (uint32_t k = 0;; ++k) {
                const uint32_t s = k % kItemRing;
                if (k >= (uint32_t)kItemRing &&
                    !wait_bar(sm, &sm.item_empty[s], ((k / kItemRing) - 1) & 1, status))
                    break;
                const Item it = find_item(p, order, round, true);
                round = it.round;
                sm.items[s] = it;
                mbar_arrive(&sm.item_full[s]);
                if (!(it.flags & 1)) break;
            }
        }
      } else {
        // ===================== dt warp (also owns the TMEM allocation) =====================
        Walker wk;
        Chunk c, cn;
        uint32_t k = 0;
        DtOut ds;
        ds.R0 = ds.R1 = 0.f;
        ds.ok = 1;
        // An item's initial state into L2 a few blocks before the state warps load it.
        auto prefetch_init = [&](const Chunk &x) {
            if (!(x.first && x.init) || lane != 0) return;
            if (x.init_ws)
                bulk_prefetch_l2(p.seg_state + (size_t)x.bin * (2 * kP * kN), 2 * kP * kN * sizeof(float));
            else
                bulk_prefetch_l2(static_cast<const StT *>(x.snap ? p.snap_states : p.state_cache) +
                                     ((int64_t)(x.snap ? x.seq : x.slot) * p.H + x.h0) * (kP * kN),
                                 2 * kP * kN * sizeof(StT));
        };
        bool have = wk.next(sm, c, false, true, status);
        if (have) prefetch_init(c);
        DtRaw dr = have ? dt_load(p, c.row0, c.l, c.h0) : DtRaw{};
        // the CTA's first block is prepared at once: the lookup of what follows
        // it may still be in flight on the item warp
        if (have) {
            ds = dt_prep(sm, p, dr, c.l, c.h0, c.first, k, ds.R0, ds.R1, status);
            ++k;
            have = ds.ok && wk.next(sm, c, false, true, status);
            if (have) prefetch_init(c);
            dr = have ? dt_load(p, c.row0, c.l, c.h0) : DtRaw{};
        }
        while (ds.ok && have) {
            const bool have_n = wk.next(sm, cn, false, true, status);
            if (have_n) prefetch_init(cn);
            const DtRaw drn = have_n ? dt_load(p, cn.row0, cn.l, cn.h0) : DtRaw{};   // next block's dt, early
            ds = dt_prep(sm, p, dr, c.l, c.h0, c.first, k, ds.R0, ds.R1, status);
            ++k;
            c = cn;
            dr = drn;
            have = have_n;
        }
      }
    } else if (warp >= 4 && warp < 8) {
        // ===================== scaled Xw (lane = token) =====================
        // Per block k, with w_s = exp(E - cum_s) dt'_s: the hi part bf16(w x) into
        // the Xw buffer once block k-1's lo MMA has read it, then the lo part
        // bf16(w x - hi) once the hi MMA has.  After each part one thread of warp
        // 4 issues that part's state MMA (hs += B^T Xw), once the state warps have
        // read hs for this block.  The four warps meet at a named barrier that
        // also ANDs their status, so they always leave the loop together.  Compact
        // loops: the hot code of all roles has to stay in the SM's instruction cache.
        const int q = warp - 4;
        const int t = q * 32 + lane;
        Walker wk;
        Chunk c;
        uint32_t kc = 0;
        bool ok = true;
        while (wk.next(sm, c, false, true, status)) {
            const uint32_t ab = kc % kArrBufs;
            const Arrays &ar = sm.arr[ab];
            const uint32_t tX = 3 * kc + 2;
            const uint8_t *xt = sm.slot[tX % kSlots];
            ok = warp_wait(sm, &sm.arr_ready[ab], (kc / kArrBufs) & 1, status) &&
                 warp_wait(sm, &sm.full[tX % kSlots], (tX / kSlots) & 1, status);
            const float w0 = (t < c.l) ? __expf(ar.E[0] - ar.cum[0][t]) * ar.dtp[0][t] : 0.f;
            const float w1 = (t < c.l) ? __expf(ar.E[1] - ar.cum[1][t]) * ar.dtp[1][t] : 0.f;
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&sm.arr_free[ab]);
            // ---- hi part bf16(w x) into the buffer once block k-1's lo MMA has read it ----
            ok = ok && (kc == 0 || warp_wait(sm, &sm.xbuf_free, 1, status));
            if (ok) {
#pragma unroll 4
            for (int i = 0; i < 16; ++i) {
                const int hh = i >> 3, cc = i & 7;
                const float2 ww = hh ? make_float2(w1, w1) : make_float2(w0, w0);
                const uint32_t off = hh * kHalfBytes + t * 128 + ((cc ^ (t & 7)) << 4);
                const uint4 xv = *reinterpret_cast<const uint4 *>(xt + off);
                uint4 o;
                o.x = pack2(__fmul2_rn(ww, make_float2(bf16_lo(xv.x), bf16_hi(xv.x))));
                o.y = pack2(__fmul2_rn(ww, make_float2(bf16_lo(xv.y), bf16_hi(xv.y))));
                o.z = pack2(__fmul2_rn(ww, make_float2(bf16_lo(xv.z), bf16_hi(xv.z))));
                o.w = pack2(__fmul2_rn(ww, make_float2(bf16_lo(xv.w), bf16_hi(xv.w))));
                *reinterpret_cast<uint4 *>(sm.xw[0] + off) = o;
            }
            }
            fence_proxy_async_smem();
            if (!xw_group_and(ok)) break;                       // hi part of all four warps in
            bool issued = true;
            if (warp == 4 && lane == 0) {
                const uint32_t tB = 3 * kc + 1;
                issued = wait_bar(sm, &sm.full[tB % kSlots], (tB / kSlots) & 1, status) &&
                         wait_bar(sm, &sm.state_ok, kc & 1, status);
                if (issued) {
                    tc_fence_after();
                    const uint64_t db = smem_desc_sw128(smem_u32(sm.slot[tB % kSlots]), kHalfBytes, 1024);
                    const uint64_t dw = smem_desc_sw128(smem_u32(sm.xw[0]), kHalfBytes, 1024);
#pragma unroll
                    for (uint32_t ks = 0; ks < 8; ++ks) mma_ss(tmem + kColH, db + ks * 128, dw + ks * 128, kIdH, 1);
                    mma_commit(&sm.xbuf_free);
                }
            }
            __syncwarp();
            // ---- lo part bf16(w x - hi) once the hi MMA has read the buffer ----
            ok = warp_wait(sm, &sm.xbuf_free, 0, status);      // fails through the abort flag if not issued
            if (ok) {
#pragma unroll 1
            for (int i = 0; i < 16; ++i) {
                const int hh = i >> 3, cc = i & 7;
                const float2 ww = hh ? make_float2(w1, w1) : make_float2(w0, w0);
                const uint32_t off = hh * kHalfBytes + t * 128 + ((cc ^ (t & 7)) << 4);
                const uint4 xv = *reinterpret_cast<const uint4 *>(xt + off);
                const uint32_t xw4[4] = {xv.x, xv.y, xv.z, xv.w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 v = __fmul2_rn(ww, make_float2(bf16_lo(xw4[e]), bf16_hi(xw4[e])));
                    const uint32_t h2 = pack2(v);
                    o[e] = pack2(__fadd2_rn(v, make_float2(-bf16_lo(h2), -bf16_hi(h2))));
                }
                *reinterpret_cast<uint4 *>(sm.xw[0] + off) = make_uint4(o[0], o[1], o[2], o[3]);
            }
            }
            fence_proxy_async_smem();
            if (!xw_group_and(ok)) break;                       // lo part of all four warps in
            if (warp == 4 && lane == 0) {
                const uint32_t tB = 3 * kc + 1;
                tc_fence_after();
                const uint64_t db = smem_desc_sw128(smem_u32(sm.slot[tB % kSlots]), kHalfBytes, 1024);
                const uint64_t dw = smem_desc_sw128(smem_u32(sm.xw[0]), kHalfBytes, 1024);
#pragma unroll
                for (uint32_t ks = 0; ks < 8; ++ks) mma_ss(tmem + kColH, db + ks * 128, dw + ks * 128, kIdH, 1);
                mma_commit(&sm.state_done);
                mma_commit(&sm.xbuf_free);
                mma_commit(&sm.empty[tB % kSlots]);
                mma_commit(&sm.empty[tX % kSlots]);          // the Xw passes have read X
            }
            __syncwarp();
            ++kc;
        }
        if (warp == 4 && lane == 0) {                          // the state MMAs' issuing thread
            mma_commit(&sm.drain_h);
            drain_wait(&sm.drain_h, 0, status);
        }
    } else if (warp >= 8 && warp < 12) {
        // ===================== S and row scaling (lane = token) =====================
        const int q = warp - 8;
        const int t = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        Walker wk;
        Chunk c;
        uint32_t kc = 0;
        bool ok = true;
        while (ok && wk.next(sm, c, false, true, status)) {
            const uint32_t ab = kc % kArrBufs;
            const Arrays &ar = sm.arr[ab];
            const uint32_t ycol = kColY + 128 * (kc & 1);
            // ---- S_h from G, in place ----
            if (!(ok = warp_wait(sm, &sm.arr_ready[ab], (kc / kArrBufs) & 1, status) &&
                       warp_wait(sm, &sm.g_ready, kc & 1, status)))
                break;
            tc_fence_after();
            const float cum_t0 = ar.cum[0][t], cum_t1 = ar.cum[1][t];
            // 16 G columns (tokens s) at a time; the 8 packed columns of each head
            // go back into the 16 just read (head h at +8h).
            // exp(cum_t - cum_s) = exp(cum_t - c_b) exp(c_b - cum_s): below the
            // diagonal 32-token block c_b is the end of the block of s (both
            // factors <= 1), on it the start (first factor <= 1, second <=
            // exp(kDiagFactorLimit)); the second factor times dt'_s is per token.
#pragma unroll 1
            for (int c16 = 0; c16 < 8; ++c16) {
                const int j = c16 >> 1;
                const uint32_t taddr = tmem + lane_off + kColG + 16 * c16;
                uint32_t out0[8], out1[8];
                if (j > q) {                                  // above the diagonal: S = 0
#pragma unroll
                    for (int i2 = 0; i2 < 8; ++i2) out0[i2] = 0u;
                    tmem_st8(taddr, out0);
                    tmem_st8(taddr + 8, out0);
                    continue;
                }
                const bool diag = (j == q);
                if (diag && (ar.exact[0][j] || ar.exact[1][j])) {
                    s_diag_exact(taddr, ar, t, c16, cum_t0, cum_t1);   // steep decay: rare
                    continue;
                }
                uint32_t g[16];
                tmem_ld16(taddr, g);
                const float b0 = diag ? (j ? ar.cumE[0][j - 1] : 0.f) : ar.cumE[0][j];
                const float b1 = diag ? (j ? ar.cumE[1][j - 1] : 0.f) : ar.cumE[1][j];
                const float *v0p = (diag ? ar.vdiag[0] : ar.vfac[0]) + 16 * c16;
                const float *v1p = (diag ? ar.vdiag[1] : ar.vfac[1]) + 16 * c16;
                const int lim = diag ? t - 16 * c16 + 1 : 16;    // causal mask: s - 16 c16 < lim
                const float u0 = __expf(cum_t0 - b0), u1 = __expf(cum_t1 - b1);
                const float2 uu0 = make_float2(u0, u0), uu1 = make_float2(u1, u1);
                tmem_wait_ld();
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    const float4 va = *reinterpret_cast<const float4 *>(v0p + 4 * i4);
                    const float4 vb = *reinterpret_cast<const float4 *>(v1p + 4 * i4);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int i2 = 2 * i4 + e;
                        const float2 gg = f2(g[2 * i2], g[2 * i2 + 1]);
                        float2 r0 = __fmul2_rn(__fmul2_rn(gg, uu0), e ? make_float2(va.z, va.w) : make_float2(va.x, va.y));
                        float2 r1 = __fmul2_rn(__fmul2_rn(gg, uu1), e ? make_float2(vb.z, vb.w) : make_float2(vb.x, vb.y));
                        const bool kx = 2 * i2 < lim, ky = 2 * i2 + 1 < lim;
                        r0.x = kx ? r0.x : 0.f;
                        r1.x = kx ? r1.x : 0.f;
                        r0.y = ky ? r0.y : 0.f;
                        r1.y = ky ? r1.y : 0.f;
                        out0[i2] = pack2(r0);
                        out1[i2] = pack2(r1);
                    }
                }
                tmem_st8(taddr, out0);
                tmem_st8(taddr + 8, out1);
            }
            tmem_wait_st();
            tc_fence_before();
            const float e0 = __expf(cum_t0), e1 = __expf(cum_t1);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.s_ready);
                mbar_arrive(&sm.arr_free[ab]);
            }
            // ---- Y[b] *= exp(cum_t) ----
            if (!(ok = warp_wait(sm, &sm.yinter_ready, kc & 1, status))) break;
            tc_fence_after();
#pragma unroll 1
            for (int c16 = 0; c16 < 8; ++c16) {
                uint32_t r[16];
                tmem_ld16(tmem + lane_off + ycol + 16 * c16, r);
                const float2 ee = (c16 >> 2) ? make_float2(e1, e1) : make_float2(e0, e0);
                tmem_wait_ld();
#pragma unroll
                for (int i2 = 0; i2 < 8; ++i2) {
                    const float2 v = __fmul2_rn(f2(r[2 * i2], r[2 * i2 + 1]), ee);
                    r[2 * i2] = __float_as_uint(v.x);
                    r[2 * i2 + 1] = __float_as_uint(v.y);
                }
                tmem_st16(tmem + lane_off + ycol + 16 * c16, r);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.y_scaled);
            ++kc;
        }
    } else if (warp >= 12) {
        // ===================== state (lane = state column n) =====================
        // The accumulator holds hs = h exp(-R).  Per block this role reads hs
        // (renormalising it when the block's scales ask for it), writes the bf16 copy of h for
        // C h^T -- warps 12-13 own n < 64, warps 14-15 n >= 64, matching the two
        // halves of that MMA -- and stores the final state of each item.  While a
        // block's state MMAs run it also writes y of the previous block (lane =
        // token there).
        const int q = warp - 12;
        const int n = q * 32 + lane;
        const bool first_half = q < 2;
        const int hrow = n & 63;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        Walker wk;
        Chunk c;
        uint32_t kc = 0;
        int32_t pend = 0;                 // 1 + state slot stored but not yet published
        // Each warp publishes its own 32 rows n of a handed-over state (the rows
        // the same warp of the next segment's CTA reads): fence, then the flag.
        auto publish = [&]() {
            __threadfence();
            __syncwarp();
            if (lane == 0 && pend - 1 != p.withhold) st_release_gpu(p.seg_flags + (size_t)(pend - 1) * 4 + q, 1);
            pend = 0;
        };
        bool ok = true;
        StT *cache = static_cast<StT *>(p.state_cache);
        StT *chunk_out = static_cast<StT *>(p.out_chunk_states);
        const bool sr = std::is_same<StT, __half>::value && p.sr_seed != nullptr;
        const uint64_t seed = sr ? *p.sr_seed : 0ull;
        int32_t prev_row0 = 0, prev_l = 0, prev_h0 = 0;   // previous block, for its y epilogue
        // y = Y + D x of block k (lane = token t here; x from the smem tile, which
        // stays until x_epi_done), run while block k+1's state MMAs execute
        auto epilogue = [&](uint32_t k) -> bool {
            const int t = n;
            const uint32_t ycol = kColY + 128 * (k & 1);
            const uint8_t *xt = sm.slot[(3 * k + 2) % kSlots];
            const bool valid = t < prev_l;
            __nv_bfloat16 *yrow = static_cast<__nv_bfloat16 *>(p.out_y) +
                                  ((int64_t)(prev_row0 + t) * p.H + prev_h0) * kP;
            const float D0 = p.D ? p.D[prev_h0] : 0.f, D1 = p.D ? p.D[prev_h0 + 1] : 0.f;
            // double buffered: block k+1's Y can be final before this check
            if (!warp_wait(sm, &sm.y_ready[k & 1], (k >> 1) & 1, status)) return false;
            tc_fence_after();
#pragma unroll 1
            for (int c16 = 0; c16 < 8; ++c16) {
                uint32_t r[16];
                tmem_ld16(tmem + lane_off + ycol + 16 * c16, r);
                const int hh = c16 >> 2;
                const float2 dd = hh ? make_float2(D1, D1) : make_float2(D0, D0);
                // x of this head and these 16 p: two 16-byte chunks of the swizzled row
                const int ch = (c16 & 3) * 2;
                const uint8_t *xrow = xt + hh * kHalfBytes + t * 128;
                const uint4 xa = *reinterpret_cast<const uint4 *>(xrow + ((ch ^ (t & 7)) << 4));
                const uint4 xb = *reinterpret_cast<const uint4 *>(xrow + (((ch + 1) ^ (t & 7)) << 4));
                tmem_wait_ld();
                if (c16 == 7) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.y_free[k & 1]);
                }
                const uint32_t xw8[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
                uint32_t yw[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    yw[e] = pack2(__ffma2_rn(dd, make_float2(bf16_lo(xw8[e]), bf16_hi(xw8[e])),
                                             f2(r[2 * e], r[2 * e + 1])));
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(yrow) + hh * 8 + ch;
                    dst[0] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
                    dst[1] = make_uint4(yw[4], yw[5], yw[6], yw[7]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.x_epi_done[k & 1]);
            return true;
        };
        while (ok && wk.next(sm, c, true, true, status)) {
            // this lane's column (+ (head*64+p)*N) of the initial state (the cache
            // slot, or its snapshot) and the element index of the final slot's
            auto init_col = [&]() {
                return (c.snap ? static_cast<const StT *>(p.snap_states) : cache) +
                       ((int64_t)(c.snap ? c.seq : c.slot) * p.H + c.h0) * (kP * kN) + n;
            };
            auto final_base = [&]() { return ((int64_t)c.fslot * p.H + c.h0) * (kP * kN) + n; };
            if (c.empty_item) {
                const StT *init_src = init_col();
                const int64_t fbase = final_base();
                if (p.write_final) {
                    for (int col = 0; col < 2 * kP; ++col) {
                        const float v = c.init ? load_state<StT>(init_src + (int64_t)col * kN) : 0.f;
                        put_state<StT>(cache, fbase + (int64_t)col * kN, v, sr, seed, 0u);
                    }
                }
                continue;
            }
            const uint32_t ab = kc % kArrBufs;
            const Arrays &ar = sm.arr[ab];
            if (!c.first) {
                if (!(ok = warp_wait(sm, &sm.arr_ready[ab], (kc / kArrBufs) & 1, status) &&
                           warp_wait(sm, &sm.state_done, (kc - 1) & 1, status)))
                    break;
                tc_fence_after();
            } else if (!c.init) {
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {             // zeros into the accumulator columns
                    uint32_t r[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) r[i] = 0u;
                    tmem_st16(tmem + lane_off + kColH + 16 * j, r);
                }
                tmem_wait_st();
            } else {
                // the item's initial state into the accumulator columns: the state
                // the previous segment's CTA handed over (possibly this CTA, its
                // publication still pending), else the cache; 64 loads in flight
                const float *ws = nullptr;
                if (c.init_ws) {
                    // publish a pending state first if this has to wait: the CTA
                    // that is to set the flag may be waiting for that one
                    const int32_t *fl = p.seg_flags + (size_t)c.bin * 4 + q;
                    if (!__all_sync(0xffffffffu, ld_acquire_gpu(fl) != 0)) {
                        if (pend) publish();
                        if (!(ok = warp_wait_flag(sm, fl, status))) break;
                    }
                    ws = p.seg_state + (size_t)c.bin * (2 * kP * kN) + n;
                }
#pragma unroll 1
                for (int j = 0; j < 2; ++j) {
                    uint32_t r[64];
                    if (ws) {
#pragma unroll
                        for (int i = 0; i < 64; ++i) r[i] = __float_as_uint(__ldcg(ws + (j * 64 + i) * kN));
                    } else {
                        const StT *init_src = init_col();
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            r[i] = __float_as_uint(load_state<StT>(init_src + (int64_t)(j * 64 + i) * kN));
                    }
                    tmem_st32(tmem + lane_off + kColH + 64 * j, *reinterpret_cast<const uint32_t(*)[32]>(r));
                    tmem_st32(tmem + lane_off + kColH + 64 * j + 32, *reinterpret_cast<const uint32_t(*)[32]>(r + 32));
                }
                tmem_wait_st();
            }
            // an item's first block: its initial state is loaded before its scales
            // are awaited (they come from the dt warp's first pass over the item)
            if (c.first && !(ok = warp_wait(sm, &sm.arr_ready[ab], (kc / kArrBufs) & 1, status))) break;
            uint32_t packed[64];                  // bf16 copy (hi part) of this lane's 128 state values
            // per head: the state entering the block is hs * eprev; renormalised
            // accumulators hold exp(dlt) h instead.  h = hi + lo with both parts
            // bf16: hi stays in registers for the two half-n copies below, lo goes
            // straight to its own buffer (row n of each head), once the previous
            // block's C h_lo^T has read it.
            const float2 ep0 = make_float2(ar.eprev[0], ar.eprev[0]), ep1 = make_float2(ar.eprev[1], ar.eprev[1]);
            const bool rn0 = ar.renorm[0] != 0, rn1 = ar.renorm[1] != 0;
            if (kc > 0 && !(ok = warp_wait(sm, &sm.hlo_free, (kc - 1) & 1, status))) break;
            uint8_t *lorow = sm.hlo[n >> 6] + hrow * 128;
            // the state entering this block ends a chunk of the sequence: store it
            // (its own pass over the accumulator, before the copies below take
            // their registers)
            const int32_t pos0 = c.row0 - c.seq_t0;
            if (chunk_out != nullptr && c.crow >= 0 && !c.first && pos0 % p.chunk_size == 0) {
                const int64_t cbase = ((int64_t)(c.crow + pos0 / p.chunk_size - 1) * p.H + c.h0) * (kP * kN) + n;
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    uint32_t r[16];
                    tmem_ld16(tmem + lane_off + kColH + 16 * j, r);
                    tmem_wait_ld();
                    const float e = (j >> 2) ? ar.eprev[1] : ar.eprev[0];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        put_state<StT>(chunk_out, cbase + (int64_t)(j * 16 + i) * kN, __uint_as_float(r[i]) * e, sr,
                                       seed, 1u);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {                 // 16 columns at a time
                uint32_t r[16];
                tmem_ld16(tmem + lane_off + kColH + 16 * j, r);
                tmem_wait_ld();
                const float2 ep = (j >> 2) ? ep1 : ep0;
                uint32_t lo[8];
#pragma unroll
                for (int i2 = 0; i2 < 8; ++i2) {     // h entering the block (eprev = 1 at an item's first block)
                    const float2 h = __fmul2_rn(f2(r[2 * i2], r[2 * i2 + 1]), ep);
                    const uint32_t hi = pack2(h);
                    packed[j * 8 + i2] = hi;
                    lo[i2] = pack2(__fadd2_rn(h, make_float2(-bf16_lo(hi), -bf16_hi(hi))));
                }
                uint8_t *lp = lorow + (j >> 2) * kHbufHead;
                const int cc = 2 * (j & 3);
                *reinterpret_cast<uint4 *>(lp + ((cc ^ (hrow & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                *reinterpret_cast<uint4 *>(lp + (((cc + 1) ^ (hrow & 7)) << 4)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
            }
            fence_proxy_async_smem();
            if (rn0 || rn1) {
                // renormalise the accumulator to exp(dlt) h (rare: the block's exponents
                // left the range of the running scale)
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    const int hh = j >> 2;
                    if (!(hh ? rn1 : rn0)) continue;
                    const float2 f = hh ? make_float2(ar.eprev[1] * ar.edlt[1], ar.eprev[1] * ar.edlt[1])
                                        : make_float2(ar.eprev[0] * ar.edlt[0], ar.eprev[0] * ar.edlt[0]);
                    uint32_t r[16];
                    tmem_ld16(tmem + lane_off + kColH + 16 * j, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i2 = 0; i2 < 8; ++i2) {
                        const float2 v = __fmul2_rn(f2(r[2 * i2], r[2 * i2 + 1]), f);
                        r[2 * i2] = __float_as_uint(v.x);
                        r[2 * i2 + 1] = __float_as_uint(v.y);
                    }
                    tmem_st16(tmem + lane_off + kColH + 16 * j, r);
                }
                tmem_wait_st();
            }
            const float2 ef0 = make_float2(ar.eend[0], ar.eend[0]), ef1 = make_float2(ar.eend[1], ar.eend[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.state_ok);
                mbar_arrive(&sm.arr_free[ab]);
                mbar_arrive(&sm.hlo_ready);
            }
            // ---- bf16 copy of h for C h^T ----
            if (first_half) {
                if (kc > 0 && !(ok = warp_wait(sm, &sm.yinter_ready, (kc - 1) & 1, status))) break;
            } else {
                if (!(ok = warp_wait(sm, &sm.hbuf_a_done, kc & 1, status))) break;
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint8_t *rowp = sm.hbuf + hh * kHbufHead + hrow * 128;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4 *>(rowp + ((cc ^ (hrow & 7)) << 4)) =
                        make_uint4(packed[hh * 32 + cc * 4], packed[hh * 32 + cc * 4 + 1],
                                   packed[hh * 32 + cc * 4 + 2], packed[hh * 32 + cc * 4 + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(first_half ? &sm.hs_a : &sm.hs_b);
            if (pend) publish();
            // ---- y of the previous block ----
            if (kc > 0 && !(ok = epilogue(kc - 1))) break;
            prev_row0 = c.row0;
            prev_l = c.l;
            prev_h0 = c.h0;
            if (c.last) {
                // final state of the item: h = hs * exp(R after the block)
                if (!(ok = warp_wait(sm, &sm.state_done, kc & 1, status))) break;
                tc_fence_after();
                if (c.fin_ws) {
                    // hand the state to the next segment: fp32 h, then the flag
                    float *ws = p.seg_state + (size_t)c.bout * (2 * kP * kN) + n;
#pragma unroll 1
                    for (int j = 0; j < 4; ++j) {
                        uint32_t r[32];
                        tmem_ld32(tmem + lane_off + kColH + 32 * j, r);
                        tmem_wait_ld();
                        const float2 ef = (j >> 1) ? ef1 : ef0;
#pragma unroll
                        for (int i2 = 0; i2 < 16; ++i2) {
                            const float2 h = __fmul2_rn(f2(r[2 * i2], r[2 * i2 + 1]), ef);
                            __stcg(ws + (j * 32 + 2 * i2) * kN, h.x);
                            __stcg(ws + (j * 32 + 2 * i2 + 1) * kN, h.y);
                        }
                    }
                    pend = c.bout + 1;            // published once the next block's h copy is out
                }
                // the item's end: the sequence's end, or a segment cut that may
                // also end a chunk
                const int32_t pos1 = c.row0 + c.l - c.seq_t0;
                const bool cend = chunk_out != nullptr && c.crow >= 0 &&
                                  (!c.fin_ws || pos1 % p.chunk_size == 0);
                const int64_t cbase_end =
                    ((int64_t)(c.crow + (pos1 - 1) / p.chunk_size) * p.H + c.h0) * (kP * kN) + n;
                const bool fin = !c.fin_ws && p.write_final;
                const int64_t fbase = final_base();
                if (fin || cend) {
#pragma unroll 1
                    for (int j = 0; j < 4; ++j) {
                        uint32_t r[32];
                        tmem_ld32(tmem + lane_off + kColH + 32 * j, r);
                        tmem_wait_ld();
                        const float2 ef = (j >> 1) ? ef1 : ef0;
#pragma unroll
                        for (int i2 = 0; i2 < 16; ++i2) {
                            const float2 h = __fmul2_rn(f2(r[2 * i2], r[2 * i2 + 1]), ef);
                            const int64_t col = j * 32 + 2 * i2;
                            if (fin) {
                                put_state<StT>(cache, fbase + col * kN, h.x, sr, seed, 0u);
                                put_state<StT>(cache, fbase + (col + 1) * kN, h.y, sr, seed, 0u);
                            }
                            if (cend) {
                                put_state<StT>(chunk_out, cbase_end + col * kN, h.x, sr, seed, 1u);
                                put_state<StT>(chunk_out, cbase_end + (col + 1) * kN, h.y, sr, seed, 1u);
                            }
                        }
                    }
                }
                tc_fence_before();
            }
            ++kc;
        }
        if (pend) publish();
        if (ok && kc > 0) epilogue(kc - 1);       // y of the last block
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
    bool prep_attr_set = false;
};
DeviceInfo g_dev[64];
std::mutex g_dev_mu;

// failure-detection test hooks (ssd_testing_set_hooks)
std::atomic<uint64_t> g_hook_wait_cycles{0};
std::atomic<int32_t> g_hook_withhold{-1};
std::atomic<int32_t> g_hook_force_unsegmented{0};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory beyond the per-CTA limit");

// Workspace: the longest-first order, then (segmentation) the level table,
// each rank's first boundary, four flags (one per state warp) and one fp32
// state per handed-over state.  `cap` states at most: no more than kSegSlots, and no more than the
// batch can have with kSegMinBlocks-block segments.
struct WsLayout {
    size_t meta = 0, bstart = 0, flags = 0, states = 0, total = 0;
    int32_t cap = 0;
};

size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

WsLayout ws_layout(int64_t T, int32_t S, int32_t H) {
    WsLayout L;
    L.total = round256((size_t)S * sizeof(int32_t));
    if (S <= 0 || S > kSortMax) return L;
    const int64_t blocks = (T + kQ - 1) / kQ + S;       // >= sum over sequences of their block counts
    const int64_t cap = std::min<int64_t>(kSegSlots, blocks * (H / 2) / kSegMinBlocks);
    if (cap <= 0) return L;
    L.cap = (int32_t)cap;
    L.meta = L.total;
    L.bstart = L.meta + round256(kMetaInts * sizeof(int32_t));
    L.flags = L.bstart + round256((size_t)S * sizeof(int32_t));
    L.states = L.flags + round256((size_t)cap * 4 * sizeof(int32_t));
    L.total = L.states + (size_t)cap * kSegStateBytes;
    return L;
}

// Segments pay off only when there are few items per SM (with more, the
// longest-first deal already balances the SMs) and the longest item is
// shorter than an SM's mean share of the work (the prep kernel decides that
// from the actual lengths).  The host rules them out beforehand -- sparing the
// cooperative launch -- when the max_seqlen hint shows that the longest item
// is at least that share even for the largest block count T and S allow, or no
// longer than the shortest segment the prep kernel would choose.  A workspace
// without room for the states (the fixed-scratch entry point) runs unsegmented.
bool may_segment(int64_t T, int32_t S, int32_t H, int32_t max_seqlen, size_t workspace_bytes, int sms) {
    const WsLayout L = ws_layout(T, S, H);
    const int64_t hp = H / 2;
    const int64_t items = (int64_t)S * hp;
    if (!(L.cap > 0 && workspace_bytes >= L.total && items > sms && items < (int64_t)kSegMaxItemsPerSm * sms))
        return false;
    if (max_seqlen > 0) {
        const int64_t nb0 = ((int64_t)max_seqlen + kQ - 1) / kQ;
        const int64_t tb = (T + kQ - 1) / kQ;
        const int64_t per = (int64_t)kSegPerSm * sms;
        const int64_t min_seg = std::max<int64_t>(kSegMinBlocks, (tb * hp + per - 1) / per);
        if (nb0 * sms >= (tb + S) * hp || nb0 <= min_seg) return false;
    }
    return true;
}

cudaError_t current_device_sms(int *sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo &di = g_dev[dev];
    if (di.sms == 0) {
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    *sms = di.sms;
    return cudaSuccess;
}

template <typename StT>
cudaError_t launch_typed(const ScanArgs &a, int st_idx, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
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
        if (!di.prep_attr_set) {
            e = cudaFuncSetAttribute(prep_order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
            if (e != cudaSuccess) return e;
            di.prep_attr_set = true;
        }
        sms = di.sms;
    }
    CUtensorMap mx, mb, mc;
    if (!make_map(&mx, a.x, (uint64_t)a.H * kP, (uint64_t)a.T) ||
        !make_map(&mb, a.B, (uint64_t)a.G * kN, (uint64_t)a.T) ||
        !make_map(&mc, a.C, (uint64_t)a.G * kN, (uint64_t)a.T))
        return cudaErrorInvalidValue;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *order = reinterpret_cast<int32_t *>(ws);
    const WsLayout L = ws_layout(a.T, a.S, a.H);
    const int hp = a.H / 2;
    const bool seg = may_segment(a.T, a.S, a.H, a.max_seqlen, workspace_bytes, sms);
    int32_t *meta = seg ? reinterpret_cast<int32_t *>(ws + L.meta) : nullptr;
    int32_t *bstart = seg ? reinterpret_cast<int32_t *>(ws + L.bstart) : nullptr;
    int32_t *flags = seg ? reinterpret_cast<int32_t *>(ws + L.flags) : nullptr;
    float *states = seg ? reinterpret_cast<float *>(ws + L.states) : nullptr;
    // Small unsegmented batches are sorted by the scan kernel itself: one launch
    // unless the initial states need a snapshot.
    const bool sort_in_cta = !seg && a.S <= kSortInCta;
    const bool snap = a.snap_flag != nullptr;
    if (!sort_in_cta || snap) {
        const SnapshotArgs sa = make_snapshot_args(a, st_idx == 0 ? SSD_F32 : st_idx == 1 ? SSD_BF16 : SSD_F16,
                                                   const_cast<int32_t *>(a.snap_flag),
                                                   const_cast<void *>(a.snap_states));
        const int pgrid = snap ? std::min(a.S, 4096) : 1;
        prep_order_kernel<<<pgrid, kPrepThreads, kPrepSmem, stream>>>(a.cu_seqlens, a.S, a.T, order, meta, bstart,
                                                                       flags, hp, sms, L.cap, seg ? 1 : 0,
                                                                       sort_in_cta ? 0 : 1, sa, snap ? 1 : 0);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
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
    p.meta = meta;
    p.bstart = bstart;
    p.seg_flags = flags;
    p.seg_state = states;
    p.seg_enabled = seg ? 1 : 0;
    p.sort_in_cta = sort_in_cta ? 1 : 0;
    p.has_init = a.has_init;
    p.state_cache = a.state_cache;
    p.out_y = a.out_y;
    p.x = a.x;
    p.device_status = a.device_status;
    p.final_slot_idx = a.final_slot_idx;
    p.slot_stride = a.slot_stride ? a.slot_stride : 1;
    p.final_slot_stride = a.final_slot_stride ? a.final_slot_stride : 1;
    p.snap_flag = a.snap_flag;
    p.snap_states = a.snap_states;
    p.out_chunk_states = a.out_chunk_states;
    p.cu_chunks = a.cu_chunks;
    p.num_chunk_rows = a.num_chunk_rows;
    p.chunk_size = a.chunk_size;
    p.sr_seed = a.sr_seed;
    const uint64_t hook_wait = g_hook_wait_cycles.load();
    p.spin_limit = hook_wait ? hook_wait : kSpinLimit;
    p.withhold = g_hook_withhold.load();
    const int grid = p.num_items < sms ? p.num_items : sms;
    if (seg && g_hook_force_unsegmented.load()) {
        // test hook: the path taken when the cooperative launch is refused
        p.seg_enabled = 0;
        chunked_scan_kernel<StT><<<grid, kThreads, kSmemBytes, stream>>>(mx, mb, mc, p);
        return cudaGetLastError();
    }
    if (!seg) {
        chunked_scan_kernel<StT><<<grid, kThreads, kSmemBytes, stream>>>(mx, mb, mc, p);
        return cudaGetLastError();
    }
    // A segment waits for the CTA that runs the previous one, so every CTA
    // must be resident at once: a cooperative launch (one CTA per SM).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, chunked_scan_kernel<StT>, mx, mb, mc, p);
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    // Fewer SMs available to this context than the grid (a partitioned GPU):
    // run every item whole instead; the prep kernel's order stays valid.
    (void)cudaGetLastError();
    p.seg_enabled = 0;
    chunked_scan_kernel<StT><<<grid, kThreads, kSmemBytes, stream>>>(mx, mb, mc, p);
    return cudaGetLastError();
}

}  // namespace

void set_test_hooks(int64_t wait_cycles, int32_t withhold, int32_t force_unsegmented) {
    g_hook_wait_cycles.store(wait_cycles > 0 ? (uint64_t)wait_cycles : 0);
    g_hook_withhold.store(withhold);
    g_hook_force_unsegmented.store(force_unsegmented ? 1 : 0);
}

bool chunked_supported(const ssd_scan_params &p) {
    if (p.io_dtype != SSD_BF16 || p.headdim != kP || p.dstate != kN) return false;
    // per-chunk states fall on 128-token block ends only
    if (p.out_chunk_states != nullptr && p.chunk_size % kQ != 0) return false;
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
    return ws_layout(p.total_tokens, p.num_seqs, p.nheads).total;
}

int32_t chunked_num_launches(const ssd_scan_params &p, size_t workspace_bytes) {
    int sms = 0;
    if (current_device_sms(&sms) != cudaSuccess) return -1;
    const bool seg = may_segment(p.total_tokens, p.num_seqs, p.nheads, p.max_seqlen, workspace_bytes, sms);
    return (!seg && p.num_seqs <= kSortInCta && !snapshot_needed(p)) ? 1 : 2;
}

cudaError_t launch_chunked(const ScanArgs &a, int state_dtype, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
    switch (state_dtype) {
        case SSD_F32: return launch_typed<float>(a, 0, workspace, workspace_bytes, stream);
        case SSD_BF16: return launch_typed<__nv_bfloat16>(a, 1, workspace, workspace_bytes, stream);
        case SSD_F16: return launch_typed<__half>(a, 2, workspace, workspace_bytes, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssd
