/*
 * fa.h -- C ABI of the GB300 (sm_103a) blocked GQA flash-attention library
 * (libfa_gb300.so).  Plain pointers and sizes only; no framework types.
 *
 * Notation ("Notation", danielwatson6.github.io/fa/fa.html):
 *   B batch, K kv heads, G query heads per kv head, T queries, S keys, H head dim.
 *
 * Layouts (all tensors dense, row-major in the order given, innermost last):
 *   q, o, dO, dq : [B, K, G, T, H]  bf16 (IEEE bfloat16 stored as uint16)
 *   k, v, dk, dv : [B, K, S, H]     bf16
 *   lse          : [B, K, G, T]     float32, natural-log logsumexp of the rows
 *   seg_q        : [B, T] int32,   seg_kv : [B, S] int32 (both or neither)
 * q arrives already multiplied by H**-0.5; the library applies no scale of its
 * own ("What is wrong with naive attention?": queries pre-scaled by H^-1/2).
 *
 * Ownership: the caller owns every buffer (device memory, 16-byte aligned, as
 * TMA requires) including the backward workspace.  The library allocates no
 * device memory, never synchronises, and enqueues all work on `stream`
 * (a cudaStream_t passed as void*; NULL = legacy default stream).
 *
 * Errors: every call validates all arguments on the host before launching
 * anything and returns one of the FA_* codes below.  A bounded device-side
 * wait that runs out of time sets a device error word; fa_check_status()
 * reports it as FA_ERR_DEVICE_TIMEOUT (and clears it).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,     /* null pointer, negative size, one seg pointer without the
                                 other, misaligned pointer, workspace too small */
  FA_ERR_UNSUPPORTED = 2,     /* H not in {64,128,256}, G not a power of two <= 128,
                                 S > 131072, B*K > 65535 */
  FA_ERR_CUDA = 3,            /* a CUDA runtime/driver call or launch failed */
  FA_ERR_DEVICE_TIMEOUT = 4   /* a bounded device wait ran out (kernel gave up) */
};

/*
 * Forward pass: for every (b, k, g, t)
 *   o[b,k,g,t,:]  = sum_s softmax_s(L)[s] * v[b,k,s,:],  L[s] = q[b,k,g,t,:] . k[b,k,s,:]
 *   lse[b,k,g,t]  = log sum_s exp(L[s])
 * over the keys kept by the mask: s <= t + (S - T) when `causal` (queries are
 * aligned to the end of the keys: for T == S this is s <= t, and the last
 * query always sees every key), and seg_q[b,t] == seg_kv[b,s] when segment ids
 * are given
 * (SegmentIds, jax_flash_attn_tpu docs: only tokens with the same id attend).
 * This is the online-softmax sweep of "Chunked attention" / "Optimizing the
 * kernel" (running max m, denominator, rescaled accumulator, output divided
 * by the denominator at the end; bf16 output from an fp32 accumulator).
 * Rows with no kept key get o = 0 and lse = -inf.  The T x S weights are never
 * written to memory and no mask array exists: masks are generated per tile
 * and tiles the mask removes entirely are skipped (axlearn PR "Optimize TPU
 * Flash Attention", lazy causal mask).
 * T and S are arbitrary (no multiple-of-128 requirement; T = 1 is a decode
 * step).  T == 0 or B*K == 0: nothing to do; S == 0: o = 0, lse = -inf.
 */
int fa_fwd(const void* q, const void* k, const void* v,
           const int32_t* seg_q, const int32_t* seg_kv, int causal,
           void* o, float* lse,
           int B, int K, int G, int T, int S, int H, void* stream);

/*
 * Split-KV forward, for few query rows per kv head (decode, T = 1, or small
 * T): the same result as fa_fwd, with every Q tile's KV-tile schedule cut
 * into n_splits contiguous slices processed by separate CTAs.  Each slice
 * writes its normalised partial output (fp32) and partial lse into
 * `workspace`; a second kernel merges them, o = sum_i exp(lse_i - lse) o_i
 * with lse = log sum_i exp(lse_i).  Not on the pages (their inference note
 * only observes that decode is memory-bound); this keeps every SM streaming
 * K and V.  n_splits in [1, 256]; 1 is fa_fwd.  `workspace` (256-byte
 * aligned) must hold fa_fwd_splitkv_workspace_size(...) bytes.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v,
                   const int32_t* seg_q, const int32_t* seg_kv, int causal,
                   void* o, float* lse, int n_splits,
                   void* workspace, size_t workspace_bytes,
                   int B, int K, int G, int T, int S, int H, void* stream);

/* Workspace bytes of fa_fwd_splitkv (0 for unsupported sizes or n_splits). */
size_t fa_fwd_splitkv_workspace_size(int B, int K, int G, int T, int S, int H, int n_splits);

/* A split count that fills one wave of the current device, floor(SMs / CTAs)
   where the Q tiles alone number fewer CTAs than SMs (1 otherwise); at most 64
   and at most the number of KV tiles. */
int fa_fwd_splitkv_default_splits(int B, int K, int G, int T, int S, int H);

/*
 * Block-sparse masks (lazy, per block): a mask over query heads is described
 * by blocks of 128 query positions x 128 keys instead of a T x S array, in the
 * spirit of splash attention's per-block mask info (MultiHeadMask /
 * process_mask, "Our first kernel" baseline).  For each mask head h (one head
 * shared by every query head, mask_heads == 1, or one per query head,
 * mask_heads == K*G with h = k*G + g) and block (qb, kb):
 *   block_class[h][qb][kb]   uint8: 0 EMPTY (skipped), 1 FULL, 2 PARTIAL
 *   partial_index[h][qb][kb] int32: index of the block's bitmask (PARTIAL)
 *   partial_bits[i][r][w]    uint32: bit j of word w = key 32*w + j of query
 *                            row r of bitmask i (128 rows x 4 words)
 * with nqb = ceil(T/128), nkb = ceil(S/128).  The mask is ANDed with the
 * causal and segment masks; all three arrays live in device memory.
 * fa_block_mask_build() fills them (host memory) from a dense host mask.
 */
int fa_fwd_masked(const void* q, const void* k, const void* v,
                  const int32_t* seg_q, const int32_t* seg_kv, int causal,
                  const uint8_t* block_class, const int32_t* partial_index,
                  const uint32_t* partial_bits, int mask_heads,
                  void* o, float* lse,
                  int B, int K, int G, int T, int S, int H, void* stream);

int fa_bwd_masked(const void* q, const void* k, const void* v,
                  const void* o, const float* lse, const void* dO,
                  const int32_t* seg_q, const int32_t* seg_kv, int causal,
                  const uint8_t* block_class, const int32_t* partial_index,
                  const uint32_t* partial_bits, int mask_heads,
                  void* dq, void* dk, void* dv,
                  void* workspace, size_t workspace_bytes,
                  int B, int K, int G, int T, int S, int H, void* stream);

/*
 * Host-side builder of the block metadata from a dense host mask
 * dense[heads][T][S] (nonzero = keep).  Writes block_class and partial_index
 * ([heads][nqb][nkb]) and up to partial_capacity bitmasks into partial_bits;
 * *n_partial receives the number of PARTIAL blocks.  Call it first with
 * partial_bits = NULL and partial_capacity = 0 to size partial_bits.
 * Returns FA_ERR_INVALID_ARG on bad arguments or too small a capacity.
 */
int fa_block_mask_build(const uint8_t* dense, int heads, int T, int S,
                        uint8_t* block_class, int32_t* partial_index,
                        uint32_t* partial_bits, int64_t partial_capacity,
                        int64_t* n_partial);

/* Bytes of device workspace fa_bwd needs for these sizes (a multiple of 256;
   0 for empty or unsupported sizes), on the current device.  Where the dK/dV
   grid (one CTA per KV tile and b*K) is smaller than the GPU, the size
   includes the split part: kernel counters and fp32 partial dK/dV tiles for up
   to 4 CTAs per KV tile.  fa_bwd runs with less, down to the D rows and the
   per-tile segment tables, but then without the Q-range split. */
size_t fa_bwd_workspace_size(int B, int K, int G, int T, int S, int H);

/*
 * Backward pass for the loss sum(o * dO): writes dq, dk, dv (bf16).
 *   P  = exp(L - lse)            (recomputed per tile from the saved lse)
 *   dP = dO . v^T,  dS = P * (dP - D),  D[b,k,g,t] = sum_h dO * o
 *   dq = dS . k,  dk = sum_g dS^T . q,  dv = sum_g P^T . dO
 * The pages give no backward; this is the textbook derivative of the forward
 * definition above.  `o` and `lse` must be those fa_fwd produced for the same
 * inputs.  `workspace` (>= fa_bwd_workspace_size bytes, 256-byte aligned)
 * holds the fp32 D rows, the per-tile segment-id ranges, one byte per KV
 * tile locating where its segment id changes (when it changes at most once)
 * and, for small grids, the split part; its contents on entry do not matter.
 * Where the dK/dV grid is smaller than the GPU, the Q tiles of each KV tile are
 * dealt to up to 4 CTAs (fa_set_bwd_q_splits).  Each stores fp32 partial dK,
 * dV.  The last of them to finish adds the partials in a fixed order, so the
 * result stays deterministic.
 * Head dims 64, 128 and 256.  H = 64 runs the H = 128 kernels: the upper 64
 * head dims of every tile arrive zero-filled (their TMA boxes lie past the
 * tensors' last dim), add nothing to S and dP, and their zero gradient rows
 * are not stored; correct, at the tensor-core cost of H = 128.
 */
int fa_bwd(const void* q, const void* k, const void* v,
           const void* o, const float* lse, const void* dO,
           const int32_t* seg_q, const int32_t* seg_kv, int causal,
           void* dq, void* dk, void* dv,
           void* workspace, size_t workspace_bytes,
           int B, int K, int G, int T, int S, int H, void* stream);

/*
 * One stage of fa_bwd, with the same arguments: stage 0 computes D and the
 * per-tile segment tables into the workspace, stage 1 writes dk and dv,
 * stage 2 writes dq.  fa_bwd runs 0, 1, 2 in that order on `stream`; stages 1
 * and 2 read only the inputs and stage 0's workspace, so a caller may run
 * them on two streams once stage 0 is done.  Returns FA_ERR_INVALID_ARG for
 * a stage outside 0..2.
 */
int fa_bwd_stage(int stage, const void* q, const void* k, const void* v,
                 const void* o, const float* lse, const void* dO,
                 const int32_t* seg_q, const int32_t* seg_kv, int causal,
                 void* dq, void* dk, void* dv,
                 void* workspace, size_t workspace_bytes,
                 int B, int K, int G, int T, int S, int H, void* stream);

/* Size of the fixed device scratch used by fa_bwd_noalloc (8 MiB). */
#define FA_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * fa_bwd without a workspace argument, for callers that cannot allocate
 * device memory themselves: for example a plugin running inside a host
 * application that owns every device allocation and offers no allocator
 * hook, or a runtime whose rules forbid allocating after start-up.  It
 * computes what fa_bwd computes and calls no cudaMalloc, cudaFree or
 * other allocating routine.  It never splits the dK/dV grid's Q ranges (the
 * partial tiles would not fit its scratch), so on grids smaller than the GPU
 * its dK and dV can differ from fa_bwd's in the last bits (fp32 summation
 * order); with that split forced off in fa_bwd (fa_set_bwd_q_splits(1)) the
 * two give the same bits.  The pages have no counterpart to this call.
 *
 * The scratch (fp32 D rows plus per-tile segment tables, the same data fa_bwd
 * keeps in its workspace) is one fixed array of FA_NOALLOC_SCRATCH_BYTES in
 * the library's device memory, present on every GPU that loads the library
 * until the process exits.  Sizes whose scratch would not fit
 * (D rows and tile tables over FA_NOALLOC_SCRATCH_BYTES, i.e. roughly
 * B*K*G*T > 2 million query rows) are rejected with FA_ERR_UNSUPPORTED before
 * anything is enqueued.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All calls
 * share the one array and every call overwrites all of the scratch it reads,
 * so nothing has to start at zero; but two calls that overlap on the GPU
 * (different streams, not ordered) race on the array and give wrong results.
 * Other arguments and status codes are those of fa_bwd.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v,
                   const void* o, const float* lse, const void* dO,
                   const int32_t* seg_q, const int32_t* seg_kv, int causal,
                   void* dq, void* dk, void* dv,
                   int B, int K, int G, int T, int S, int H, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns FA_OK, FA_ERR_DEVICE_TIMEOUT or FA_ERR_CUDA.
 */
int fa_check_status(void* stream);

/* Static, NUL-terminated description of a status code. */
const char* fa_status_string(int status);

/*
 * Time limit, in nanoseconds, of every bounded device wait launched after
 * this call (default 2e9, or the FA_WAIT_LIMIT_NS environment variable).
 * Returns FA_ERR_INVALID_ARG for 0.
 */
int fa_set_wait_limit_ns(uint64_t ns);

/*
 * Keys per KV tile of the backward kernels for H <= 128 calls made after this
 * one: 0 (default) chooses per call (128, or 64 when the dK/dV grid of
 * ceil(S/128)*B*K CTAs would not fill the GPU), 64 or 128 force that size.
 * H = 256 always uses 64.  The result does not depend on the choice beyond
 * fp32 summation order.  Returns FA_ERR_INVALID_ARG for any other value.
 */
int fa_set_bwd_kv_rows(int rows);

/*
 * Q-range split of the dK/dV grid, for backward calls made after this one:
 * 0 (default) chooses per call, 1..4 forces that many CTAs per KV tile.  Either
 * applies only where the dK/dV grid is smaller than the GPU and the workspace
 * holds the split part (fa_bwd_workspace_size); elsewhere there is one CTA per
 * KV tile.  The default, for H <= 128, is the largest count in 1..4 that keeps
 * the split grid to one wave; for H = 256, the count that minimises (waves of
 * the split grid) / count, ties going to the larger count for causal,
 * segment-id or block-masked calls (uneven sweeps) and to the smaller
 * otherwise.  The result
 * does not depend on the choice beyond fp32 summation order.  Returns
 * FA_ERR_INVALID_ARG for any other value.
 */
int fa_set_bwd_q_splits(int n);

/*
 * The backward's grid plan with the default knobs, on a GPU with sm_count SMs,
 * for the shapes of an fa_bwd (masked != 0: segment ids or a block mask are
 * given): *kv_rows = keys per KV tile (64 or 128), *q_splits = CTAs per KV tile
 * of the dK/dV grid (1-4; used where the workspace holds the split part).  A
 * host-only query: touches no device.  Returns FA_ERR_INVALID_ARG for null
 * outputs or a negative sm_count, and the shape errors of fa_bwd.
 */
int fa_bwd_plan(int B, int K, int G, int T, int S, int H, int causal, int masked,
                int sm_count, int* kv_rows, int* q_splits);

/*
 * Forward grid for calls made after this one: 0 (default) chooses per call, 1
 * launches one CTA per Q tile, 2 launches one persistent CTA per SM that walks
 * the Q tiles, the next tile's schedule, Q copy and first products overlapping
 * the current tile's epilogue (H <= 128 without split-KV; other calls use one
 * CTA per Q tile).  The default takes 2 where supported and the Q tiles
 * outnumber the SMs.  The results do not depend on the choice.  Returns
 * FA_ERR_INVALID_ARG for any other value.
 */
int fa_set_fwd_schedule(int mode);

/*
 * Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier no one arrives on, with the current limit, and returns the status
 * fa_check_status() reports afterwards (FA_ERR_DEVICE_TIMEOUT when the
 * machinery works).  Faults nothing and leaves the context usable.
 */
int fa_selftest_wait_timeout(void* stream);

/* Number of SMs of the current device (0 on error); used for grid sizing. */
int fa_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
