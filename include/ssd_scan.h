/*
 * ssd_scan.h -- C ABI of the GB300 (sm_103a) Mamba2 SSD varlen scan library.
 *
 * The operation (one call = one Mamba2 layer's SSD scan over a packed batch):
 * the chunked SSD scan of Mamba2 prefill, continued prefill and MTP
 * verification.  The pages run it as five Triton launches (cumsum, chunk
 * state, state passing, bmm, chunk scan) or as FlashInfer's fused two-launch
 * scan over packed cu_seqlens (vLLM PR #61501 "Details"); initial states are
 * read straight from the cache slot instead of a dense gather (vLLM PR #62922
 * "Details"); final states are written back in the cache dtype (vLLM PR
 * #61501 "Details"); MTP keeps the state after every speculative token (vLLM
 * PR #52928 "Summary").  The pages do not print the recurrence; this library
 * computes, for sequence s = tokens cu_seqlens[s] .. cu_seqlens[s+1]-1 and
 * head h (group g = h / (nheads / ngroups)):
 *
 *   dt'_t    = softplus(dt[t,h] + dt_bias[h])      if dt_softplus
 *            = dt[t,h] + dt_bias[h]                 otherwise (bias 0 if NULL)
 *   h_{-1}   = has_init[s] ? state_cache[slot_idx[s], h] : 0   (fp32 math)
 *   h_t[p,n] = exp(dt'_t A[h]) h_{t-1}[p,n] + dt'_t x[t,h,p] B[t,g,n]
 *   y[t,h,p] = sum_n C[t,g,n] h_t[p,n] + D[h] x[t,h,p]          (D 0 if NULL)
 *   state_cache[final_slot[s], h] = h_last (write_final; final_slot = slot_idx
 *                                           unless final_slot_idx is given;
 *                                           rounded to nearest even in the
 *                                           cache dtype, or stochastically, see
 *                                           sr_seed)
 *   out_intermediate[t, h] = h_t           (if not NULL)
 *   out_chunk_states[cu_chunks[s] + c, h] = h after token
 *       min((c + 1) chunk_size, len_s) - 1 of sequence s  (if not NULL): the
 *       state at every chunk boundary, which prefills that store Mamba
 *       checkpoints need (vLLM PR #61501 "Details")
 *
 * Layouts (all dense, row-major, innermost index last):
 *   x, out_y         [T, H, P]            io_dtype (F32 or BF16)
 *   B, C             [T, G, N]            io_dtype
 *   dt               [T, H]               float32 (raw, before bias/softplus)
 *   dt_bias, A, D    [H]                  float32 (dt_bias, D may be NULL)
 *   cu_seqlens       [S+1]                int32, device; cu[0] = 0, cu[S] = T,
 *                                         non-decreasing (empty sequences ok)
 *   state_cache      [num_slots, H, P, N] state_dtype (F32, BF16 or F16)
 *   slot_idx         [S]                  int32, device, entry s at
 *                                         slot_idx[s * slot_idx_stride]
 *   final_slot_idx   [S]                  int32, device, or NULL (= slot_idx)
 *   has_init         [S]                  uint8, device, or NULL (= all zero)
 *   out_intermediate [T, H, P, N]         state_dtype, or NULL
 *   out_chunk_states [num_chunk_rows, H, P, N] state_dtype, or NULL
 *   cu_chunks        [S+1]                int32, device: cu_chunks[0] = 0 and
 *                                         cu_chunks[s+1] - cu_chunks[s] =
 *                                         ceil(len_s / chunk_size)
 * All pointers except `workspace` may be any device-accessible pointer the
 * kernels can read; the library itself never dereferences them on the host.
 *
 * Ownership: the caller owns every buffer.  The library allocates nothing,
 * frees nothing and never synchronises: a call validates its arguments on
 * the host, enqueues at most two kernels on `stream` and returns.  Nothing is
 * read back to the host, so a call may be captured in a CUDA graph.  A batch
 * the tensor-core path cuts into segments is launched cooperatively (its CTAs
 * hand states to one another); where the context has fewer SMs than the
 * device, that launch falls back to running every sequence whole.
 *
 * Aliasing and snapshot semantics: state_cache is read (initial states) and
 * written (final states) in place; by default a sequence's final state goes
 * into the slot its initial state came from, and final_slot_idx sends it
 * elsewhere.  Every initial state is the slot's content from before the call,
 * even when another sequence of the same call writes that slot (crossed or
 * shared slots; vLLM PR #62922 "Details": multi-sequence calls keep snapshot
 * semantics).  The library takes that snapshot itself: when has_init and
 * write_final are set for more than one sequence, a pass before the scan
 * copies every initial state that another sequence's final slot would
 * overwrite into the workspace (counted by ssd_scan_varlen_workspace_size).
 * A caller that knows no slot is both read by one sequence and written by
 * another sets slots_disjoint = 1 to skip that pass.  Two sequences that
 * write the same final slot leave one of the two final states there
 * (unspecified which).  out_y, out_intermediate and out_chunk_states must not
 * overlap any input.  Slots named neither by slot_idx nor final_slot_idx are
 * never read or written.
 *
 * Errors: invalid arguments return an error status and launch nothing.
 * Metadata that can only be checked on the device (slot index outside
 * [0, num_slots), cu_seqlens out of range or decreasing) makes the kernels
 * skip that sequence and OR a flag into *device_status (if not NULL); the
 * kernels never trap.
 */
#ifndef SSD_SCAN_H_
#define SSD_SCAN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* = cudaStream_t */

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,  /* bad size, NULL required pointer, bad dtype */
    SSD_ERR_UNSUPPORTED = 2,  /* valid but not compiled (e.g. dstate > 256) */
    SSD_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than required   */
    SSD_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed          */
    SSD_ERR_SCRATCH_LIMIT = 5 /* batch larger than the fixed scratch of
                                 ssd_scan_varlen_noalloc                    */
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1, SSD_F16 = 2 } ssd_dtype;

/* bits OR-ed into *device_status by the kernels */
#define SSD_DEV_BAD_SLOT 1        /* slot_idx[s] outside [0, num_slots)        */
#define SSD_DEV_BAD_SEQLENS 2     /* cu_seqlens[s..s+1] not within [0, T]      */
#define SSD_DEV_TIMEOUT 4         /* an internal wait of the chunked kernel ran
                                     out of time; its outputs are incomplete   */
#define SSD_DEV_BAD_CHUNKS 8      /* cu_chunks does not match the sequence
                                     lengths or num_chunk_rows: that
                                     sequence's chunk states are not written  */
#define SSD_DEV_BAD_RING 16       /* ssd_replay_mtp: ring_start / ring_count out
                                     of range, or the window does not fit the
                                     ring; that request is skipped             */

typedef struct {
    int64_t total_tokens;       /* T                                          */
    int32_t num_seqs;           /* S                                          */
    int32_t max_seqlen;         /* host hint, >= every sequence length, or 0
                                   when unknown; only selects the kernel      */
    int32_t nheads;             /* H                                          */
    int32_t headdim;            /* P                                          */
    int32_t dstate;             /* N                                          */
    int32_t ngroups;            /* G, divides H                               */
    int32_t chunk_size;         /* >= 1: the spacing of out_chunk_states;
                                   y and final states do not depend on it
                                   beyond rounding                            */
    int32_t io_dtype;           /* ssd_dtype of x, B, C, out_y                */
    int32_t state_dtype;        /* ssd_dtype of state_cache, out_intermediate */
    int32_t dt_softplus;        /* 1: dt' = softplus(dt + dt_bias)            */
    int32_t write_final;        /* 1: write h_last into state_cache[slot]    */
    int32_t num_slots;          /* rows of state_cache                        */
    int32_t reserved0;
    const void *x;
    const float *dt;
    const float *dt_bias;       /* may be NULL                                */
    const float *A;
    const void *B;
    const void *C;
    const float *D;             /* may be NULL                                */
    const int32_t *cu_seqlens;
    void *state_cache;          /* may be NULL only if no sequence reads or
                                   writes a slot (has_init NULL, no final)    */
    const int32_t *slot_idx;    /* may be NULL under the same condition       */
    const uint8_t *has_init;    /* may be NULL                                */
    void *out_y;
    void *out_intermediate;     /* may be NULL                                */
    void *workspace;            /* device scratch, see workspace_size         */
    size_t workspace_bytes;
    int32_t *device_status;     /* device int32 or NULL                       */
    /* ---- optional parts of a call: zero / NULL turns each off ---- */
    void *out_chunk_states;     /* per-chunk states, see the layout above     */
    const int32_t *cu_chunks;   /* required with out_chunk_states             */
    int32_t num_chunk_rows;     /* rows of out_chunk_states                   */
    int32_t slots_disjoint;     /* 1: no slot is read by one sequence and
                                   written by another (no snapshot pass)      */
    const int32_t *final_slot_idx;   /* see above                             */
    int64_t slot_idx_stride;         /* elements between entries, 0 = 1       */
    int64_t final_slot_idx_stride;   /* elements between entries, 0 = 1       */
    const uint64_t *sr_seed;    /* device, or NULL.  With state_dtype F16,
                                   final and chunk states are rounded
                                   stochastically: element e (flat index in
                                   its tensor) rounds away from zero with
                                   probability f = (|v| - |lo|) / (|hi| - |lo|)
                                   (lo, hi: the fp16 values around v toward
                                   and away from zero), i.e. when f * 2^32 >
                                   word (e & 3) of Philox4x32-10 with key
                                   (seed, seed >> 32) and counter (e >> 2,
                                   e >> 34, stream, 0); stream 0 for
                                   state_cache, 1 for out_chunk_states (vLLM
                                   PR #61501 "Details": the ReplaySSM Philox
                                   seed, read from a device buffer).  Ignored
                                   for other state dtypes.                    */
} ssd_scan_params;

/* Bytes of device workspace a call with these parameters needs (a function
 * of T, S, H and the selected kernel only; may be 0).  The workspace must be
 * 256-byte aligned and is overwritten by the call.  On the tensor-core path it
 * holds the longest-first sequence order and, for batches whose work is spread
 * over several SMs per sequence, the fp32 states that segments of one sequence
 * hand to each other (at most 1024 x 64 KiB).  Returns 0 for invalid
 * parameters as well; ssd_scan_varlen reports those. */
size_t ssd_scan_varlen_workspace_size(const ssd_scan_params *params);

/* Enqueue the scan on `stream` (NULL = legacy default stream): the SSD
 * recurrence above over every packed sequence of cu_seqlens (vLLM PR #61501
 * "Details": one varlen scan of the packed batch), initial states read from
 * their cache slots with snapshot semantics (vLLM PR #62922 "Details") and
 * final, per-token or per-chunk states written in the cache dtype (vLLM PR
 * #61501 "Details").  Returns SSD_OK when the kernels were enqueued; invalid
 * arguments come back as SSD_ERR_* with nothing enqueued, launch errors as
 * SSD_ERR_CUDA, and faults in device-resident inputs (slots, lengths, chunk
 * rows) as bits of *device_status.  Never synchronises. */
ssd_status ssd_scan_varlen(const ssd_scan_params *params, struct CUstream_st *stream);

/* Number of kernels a call with these parameters launches (the pages' path
 * takes five Triton launches, vLLM PR #61501 "Details"): 0 for an empty
 * batch, else 1 or 2 (the tensor-core path sorts a batch of at most 32
 * sequences that it does not cut into segments inside its one kernel; the
 * choice depends on params->workspace_bytes and the current device's SM
 * count).  -1 if the parameters are invalid or the device query fails. */
int32_t ssd_scan_varlen_num_launches(const ssd_scan_params *params);

/* Name of the kernel path a call would take: "chunked_tc" (tcgen05 chunked
 * scan), "recurrent" (token-by-token SIMT scan: fp32 I/O, intermediate
 * states, continuations of at most 3 tokens -- the MTP verification shape of
 * vLLM PR #52928 "Summary" -- other shapes) or "invalid". */
const char *ssd_scan_varlen_path(const ssd_scan_params *params);

/* Maximum number of sequences ssd_scan_varlen_noalloc accepts on the
 * tensor-core path. */
#define SSD_NOALLOC_MAX_SEQS 65536

/* The same scan as ssd_scan_varlen for callers that cannot allocate device
 * memory (the pages have no counterpart: this is a library convenience).
 * Examples: an engine that hands all free HBM to its state and KV pools and
 * allows no later cudaMalloc, a plug-in ABI that only passes the caller's own
 * tensors, or a latency-critical path that cannot afford cudaMalloc's
 * device-wide synchronisation.  Instead of params->workspace (ignored here)
 * the scratch comes from a fixed array in the library's device memory, so
 * the call allocates nothing and calls no allocating routine (the first call
 * on a device may load the library's module, which places the array; callers
 * that reserve all free memory should make one call before doing so).
 *   - Limit: on the tensor-core path num_seqs <= SSD_NOALLOC_MAX_SEQS, else
 *     SSD_ERR_SCRATCH_LIMIT and nothing is enqueued (the token-by-token path
 *     uses no scratch).  Calls that need the snapshot of initial states
 *     (several sequences with has_init and write_final, slots_disjoint = 0)
 *     are rejected the same way: the array has no room for states.  Every GPU
 *     that loads the library keeps the array (256 KiB) until the process exits.
 *   - Each call looks up the array's device address with the call's device
 *     current; the first lookup on a device may load the module, so make the
 *     first call before any stream capture.
 *   - All calls share the array.  Calls whose kernels may overlap on the GPU
 *     (unordered streams) race on it; order them on one stream or use
 *     ssd_scan_varlen with separate workspaces.  Nothing in the array needs
 *     to start zeroed: each call rewrites what it reads.
 *   - Every sequence runs whole on one CTA (the array has no room for the
 *     hand-over states), so for batches that ssd_scan_varlen cuts into
 *     segments the results agree with it within rounding, not bit for bit,
 *     and take longer.  ssd_scan_varlen_num_launches called with
 *     workspace_bytes = 0 gives this entry point's launch count.
 * Everything else (arguments, aliasing, errors, results) is as for
 * ssd_scan_varlen. */
ssd_status ssd_scan_varlen_noalloc(const ssd_scan_params *params, struct CUstream_st *stream);

/* ReplaySSM-style multi-token verification (vLLM PR #52928 "Summary": each
 * layer keeps a checkpoint and a ring of inputs; the accepted length advances
 * a shared cursor before the next forward; the checkpoint is updated only
 * when the next verification window would overflow the ring).  Instead of
 * storing the state after every speculative token, request s keeps, in slot
 * q = slot_idx[s]:
 *   state_cache[q]          the checkpoint,
 *   ring_x/ring_dt/ring_B[q] the raw inputs (x, dt before bias/softplus, B)
 *                           of the accepted tokens since the checkpoint, at
 *                           positions (ring_start[s] + j) mod ring_capacity,
 *                           j < ring_count[s].
 * One call, with the window tokens of every request packed by cu_seqlens:
 *   1. h = checkpoint advanced through the ring_count[s] pending inputs;
 *   2. if ring_count[s] + window length > ring_window, the checkpoint becomes
 *      h (cache dtype; stochastic rounding as in ssd_scan_params.sr_seed);
 *   3. y of every window token from h, exactly as ssd_scan_varlen computes it;
 *   4. the window's raw inputs are written to the ring positions following
 *      the pending ones;
 *   5. ring_start_out[s] / ring_count_out[s] receive where the live part of
 *      the ring now starts and how many entries precede the window (after a
 *      fold: the window's position and 0; else ring_start[s], ring_count[s]).
 *      After sampling, the caller sets ring_start = ring_start_out and
 *      ring_count = ring_count_out + accepted tokens.
 * Requirements: ring_capacity >= ring_window + every window length (the
 * window then never overwrites a pending entry); 0 <= ring_count <=
 * ring_window; distinct slots per call; the scan fields write_final,
 * out_intermediate, out_chunk_states and final_slot_idx unused (0 / NULL);
 * has_init ignored (the checkpoint is always read).  Violations found on the
 * device set SSD_DEV_BAD_RING and skip the request.  Layouts (dense):
 *   ring_x [num_slots, ring_capacity, H, P]  io_dtype
 *   ring_dt [num_slots, ring_capacity, H]    float32
 *   ring_B [num_slots, ring_capacity, G, N]  io_dtype
 * One kernel launch; no workspace; nothing is allocated or synchronised. */
typedef struct {
    ssd_scan_params scan;       /* window tokens, layer parameters, checkpoints */
    void *ring_x;
    float *ring_dt;
    void *ring_B;
    int32_t ring_capacity;
    int32_t ring_window;
    const int32_t *ring_start;  /* device [S] */
    const int32_t *ring_count;  /* device [S] */
    int32_t *ring_start_out;    /* device [S], must not alias ring_start */
    int32_t *ring_count_out;    /* device [S], must not alias ring_count */
} ssd_replay_params;

ssd_status ssd_replay_mtp(const ssd_replay_params *params, struct CUstream_st *stream);

/* Static description of a status code. */
const char *ssd_status_string(ssd_status status);

/* Test hooks of the tensor-core kernel's failure detection, for tests only
 * (process-wide; restore with (0, -1, 0)).  No page counterpart.
 *   wait_cycles > 0: every internal wait gives up after that many clock cycles
 *     instead of about two seconds, sets SSD_DEV_TIMEOUT and makes the CTA's
 *     roles leave their loops (the CTA still waits for its own TMA loads and
 *     MMAs and frees its tensor memory before it exits);
 *   withhold_handover >= 0: the segment hand-over with that index (boundary x
 *     head pairs + head pair, in the order the prep kernel numbers them) is
 *     never published, so the segment waiting for it runs out of time: the
 *     host-made fault of the failure-detection test;
 *   force_unsegmented = 1: batches that would be cut into segments run every
 *     sequence whole instead (the path taken when a cooperative launch is
 *     refused). */
void ssd_testing_set_hooks(int64_t wait_cycles, int32_t withhold_handover, int32_t force_unsegmented);

#ifdef __cplusplus
}
#endif

#endif /* SSD_SCAN_H_ */
