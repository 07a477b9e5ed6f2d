/*
 * attn_slice.h -- C ABI of a GB300 (sm_103a) masked-attention forward.
 *
 * Three operations, all enqueued on the caller's CUDA stream:
 *
 *   attn_build_tiles  slice list -> tile metadata with CSR key-tile lists
 *   attn_fwd          O = softmax(scale * Q K^T + mask) V and the row LSE
 *   attn_merge        exact combination of KV-split partial (O, lse) pairs
 *
 * Sources (web pages on flexible-mask / block-sparse attention):
 *   - MagiAttention v1.1.0 release page (xinfinite.net, "Blackwell adaptation"
 *     bullets): flexible masks as slices, an efficient block-sparse mask
 *     generation operator that never materialises the full mask, CSR
 *     compression of the mask metadata, register-to-predicate boundary checks,
 *     a thin launch path.
 *   - UltraAttn blog page (blog.ulna520.top), section 3: Full / Causal / Empty
 *     blocks of the two-dimensional attention matrix, Empty blocks skipped;
 *     section 3.2: per-KV-shard summaries (m, l, o) merged by the global max.
 *   - FlashAttention-4 news page (163.com): conditional softmax rescaling and
 *     the asynchronous MMA + tensor-memory pipeline on Blackwell.
 *
 * Conventions
 *   - No call allocates device memory: the caller owns every buffer.
 *   - Pointers named d_* / q, k, v, out, lse are device pointers; h_* are host.
 *   - Every call returns ATTN_OK (0) or an ATTN_ERR_* code.  Argument errors
 *     are found on the host before anything is launched.  Errors raised inside
 *     a kernel (a bounded wait that ran out, metadata capacity) are recorded on
 *     the device and returned by attn_last_device_error().
 *   - Calls are asynchronous with respect to the host unless stated.
 *   - Layouts (row-major, elements contiguous in the last index):
 *       Q   [S_q, H,   d] bf16        K, V [S_k, H_k, d] bf16
 *       O   [S_q, H,   d] bf16 or f32 lse  [H, S_q] f32 (natural log)
 *     All of q, k, v, out must be 16-byte aligned; they must not alias out.
 */
#ifndef ATTN_SLICE_H
#define ATTN_SLICE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (0 = the legacy default stream). */
typedef struct CUstream_st *attn_stream_t;

/* ---- status codes ------------------------------------------------------ */
#define ATTN_OK              0
#define ATTN_ERR_INVALID_ARG 1  /* bad size, range, type, null pointer        */
#define ATTN_ERR_OVERLAP     2  /* two slices' rectangles intersect            */
#define ATTN_ERR_UNSUPPORTED 3  /* head dim, tile shape, alignment not served  */
#define ATTN_ERR_CAPACITY    4  /* workspace too small for the metadata        */
#define ATTN_ERR_CUDA        5  /* a CUDA runtime call failed                  */
#define ATTN_ERR_TIMEOUT     6  /* a bounded device wait ran out (no hang)     */

/* ---- mask slice kinds ----------------------------------------------------
 * Local coordinates a = i - q_start, b = j - k_start, L_q = q_end - q_start,
 * L_k = k_end - k_start.  The pages name these kinds without defining them;
 * the reading used here is:
 *   FULL        every (i, j) of the rectangle
 *   CAUSAL      b <= a + (L_k - L_q)     bottom-right aligned
 *   INV_CAUSAL  b >= a                   top-left aligned
 *   BI_CAUSAL   both                                                          */
#define ATTN_MASK_FULL       0
#define ATTN_MASK_CAUSAL     1
#define ATTN_MASK_INV_CAUSAL 2
#define ATTN_MASK_BI_CAUSAL  3

/* ---- tile kinds (UltraAttn page, section 3: Full / Causal / Empty) ------- */
#define ATTN_TILE_FULL   1   /* every pair valid: no per-element mask       */
#define ATTN_TILE_MASKED 2   /* some pairs valid: masked from slice refs    */
                             /* Empty tiles have no entry at all            */
/* ---- block-grid kinds (attn_slices_from_block_grid input; UltraAttn page,
 * section 3: a block is Full when every position is valid, Causal when the
 * positions on and below its diagonal are, Empty when none is) ----------- */
#define ATTN_GRID_EMPTY  0
#define ATTN_GRID_FULL   1
#define ATTN_GRID_CAUSAL 2

/* ---- element types ------------------------------------------------------ */
#define ATTN_DTYPE_BF16 0
#define ATTN_DTYPE_F32  1

/* Forward kernel tile shapes: 256 query rows (two 128-row MMA tiles) by 128
 * keys for the single-CTA kernel; 512 query rows by 128 keys (head dim 128)
 * selects the CTA-pair kernel, in which two CTAs of a cluster share each
 * M = 256 MMA and each loads half of every K/V tile (FlashAttention-4 page,
 * 2-CTA MMA).  attn_fwd requires tiles built with one of these shapes. */
#define ATTN_FWD_TILE_Q 256
#define ATTN_FWD_PAIR_TILE_Q 512
#define ATTN_FWD_TILE_K 128
#define ATTN_MERGE_MAX_PARTS 16

/* One mask slice, half-open ranges [q_start, q_end) x [k_start, k_end). */
typedef struct {
  int32_t q_start, q_end, k_start, k_end, type;
} attn_slice_t;

/* Tile metadata.  Filled by attn_build_tiles; every pointer points into the
 * caller's workspace on the device and stays valid while it lives.  The
 * status word totals[3] is ATTN_OK once the build has finished normally;
 * attn_fwd and attn_bwd read it on the device and refuse metadata whose
 * status is anything else (see attn_last_device_error).
 *   row_ptr [n_qtiles+1]  CSR row pointers over query tiles
 *   col_idx [nnz]         key-tile index, ascending within a query tile
 *   kind    [nnz]         ATTN_TILE_FULL or ATTN_TILE_MASKED
 *   pairs   [nnz]         exact number of valid (query, key) pairs in the tile
 *   ref_ptr [nnz+1]       entry e uses ref_idx[ref_ptr[e] .. ref_ptr[e+1])
 *   ref_idx [nref]        ids of the slices with valid pairs in a MASKED tile,
 *                         ascending; FULL tiles reference none
 *   sched   [n_qtiles]    query tiles by descending entry count, ties by
 *                         ascending index (longest-processing-time order)
 *   totals  [4]           nnz, nref, total valid pairs, device status code
 *   slices  [n_slices]    device copy of the slice list                   */
typedef struct {
  int32_t sq, sk, tile_q, tile_k, n_qtiles, n_ktiles, n_slices, reserved;
  int64_t cap_entries, cap_refs;
  int32_t *row_ptr, *col_idx, *pairs, *ref_ptr, *ref_idx, *sched;
  uint8_t *kind;
  int64_t *totals;
  attn_slice_t *slices;
  int32_t *scratch;      /* per-query-tile counters used while building */
} attn_tiles_t;

/* Workspace needed by attn_build_tiles for this slice list (host call, no
 * device work).  The bound counts, per slice, the tiles its rectangle
 * touches, so it never undercounts.  Errors: INVALID_ARG on a bad size or
 * slice (same checks as attn_build_tiles, without the overlap test). */
int attn_tiles_workspace_bytes(const attn_slice_t *h_slices, int n_slices, int sq, int sk,
                               int tile_q, int tile_k, size_t *bytes);

/* Slice list -> tile metadata (MagiAttention page: block-sparse mask
 * generation without materialising the mask, CSR-compressed metadata;
 * UltraAttn page, section 3: Full / Causal / Empty tiles).
 *   h_slices   host array of n_slices slices (n_slices >= 0; empty slices
 *              are allowed and ignored); must be pairwise disjoint
 *   sq, sk     query / key sequence lengths (>= 1)
 *   tile_q/k   tile shape, 1..1024 each; ceil(sk / tile_k) <= 8192
 *   d_ws       device workspace of ws_bytes >= attn_tiles_workspace_bytes()
 *   tiles      host struct, filled with the shape and device pointers
 * The slice list is read on the host during the call.  The call copies it,
 * with the per-query-tile slice lists it derives, into an input image of its
 * own, so h_slices may be reused or freed as soon as the call returns.  Up to
 * 2 KB, the image travels in the build kernel's launch parameters; a larger
 * one is copied to the start of d_ws (cudaMemcpyAsync on `stream`).  The
 * metadata is produced on `stream` by one cooperative kernel when every query
 * tile's CTA fits on the GPU at once, else by two kernels.  The counts are
 * exact integers, so the result is bit-identical run to run.  The cooperative
 * kernel's grid-wide barrier is a bounded wait (attn_set_wait_limit_ns); if it
 * runs out, every query tile gets an empty list, totals[0..2] are 0, totals[3]
 * is ATTN_ERR_TIMEOUT and attn_last_device_error() reports TIMEOUT: the
 * metadata stays safe to read and the kernels that use it refuse it.
 * Errors: INVALID_ARG, OVERLAP, UNSUPPORTED (tile or grid too large),
 * CAPACITY (ws_bytes too small), CUDA. */
int attn_build_tiles(const attn_slice_t *h_slices, int n_slices, int sq, int sk,
                     int tile_q, int tile_k, void *d_ws, size_t ws_bytes,
                     attn_tiles_t *tiles, attn_stream_t stream);

/* attn_build_tiles without any device memory from the caller beyond the
 * input slice list and the output buffer.  The pages have no counterpart: it
 * exists for callers that cannot allocate, or lend, scratch memory at the
 * moment they build a mask -- for example a serving process whose device
 * memory is handed out by its own pool fixed at start-up, or a plugin inside
 * another framework that only receives pre-sized input and output buffers.
 * The per-query-tile counters that attn_build_tiles keeps in the caller's
 * workspace live instead in one fixed array inside this library
 * (ATTN_NOALLOC_MAX_QTILES entries, 20 bytes each, 320 KiB), which every GPU
 * that loads the library holds until the process exits.
 *   arguments   as attn_build_tiles; d_out (256-byte aligned) receives the
 *               metadata and needs out_bytes >= attn_tiles_workspace_bytes():
 *               the same size as attn_build_tiles' workspace, since the
 *               metadata keeps that layout (its four counter regions are
 *               simply left unused); only the counters move into the
 *               library's array
 *   limits      ceil(sq / tile_q) <= ATTN_NOALLOC_MAX_QTILES, else CAPACITY
 * No cudaMalloc, cudaFree or other allocating call is made.  The first call
 * on a device looks up the array's device address once (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture.
 * All calls share the one array, which keeps the last call's contents (the
 * kernels overwrite every counter they read, so nothing needs clearing):
 * calls whose work overlaps on the GPU -- on different streams, or from
 * different threads -- race on it and must be serialised by the caller.
 * Errors: as attn_build_tiles. */
#define ATTN_NOALLOC_MAX_QTILES 16384
int attn_build_tiles_noalloc(const attn_slice_t *h_slices, int n_slices, int sq, int sk,
                             int tile_q, int tile_k, void *d_out, size_t out_bytes,
                             attn_tiles_t *tiles, attn_stream_t stream);

/* Copies totals[0..3] (nnz, nref, total valid pairs, status) to the host;
 * synchronises `stream` first. */
int attn_tiles_totals(const attn_tiles_t *tiles, int64_t h_totals[4], attn_stream_t stream);

/* Full / Causal / Empty block grid -> slice list (host only).  UltraAttn
 * page, section 3: the attention matrix cut into (query chunk x key chunk)
 * blocks, each Full (every position valid), Causal (only part valid: here
 * the positions on and below the block's diagonal) or Empty (skipped).  One
 * slice per non-Empty block, in row-major block order: FULL -> a full slice
 * of the block, CAUSAL -> a causal slice of the block (requires
 * block_q == block_k).
 *   h_grid     uint8 [nbq * nbk] of ATTN_GRID_*
 *   h_out      room for `capacity` slices; *n_out receives the count
 * Errors: INVALID_ARG (bad kind, causal on a non-square block), CAPACITY. */
int attn_slices_from_block_grid(const uint8_t *h_grid, int nbq, int nbk, int block_q, int block_k,
                                attn_slice_t *h_out, int capacity, int *n_out);

/* Masked attention forward (UltraAttn page, section 3.3: for a fixed query
 * tile merge over its valid KV tiles, skip Empty ones; FlashAttention-4 page:
 * asynchronous MMA with tensor-memory accumulators, conditional rescaling).
 *   q, k, v     bf16 device tensors in the layouts above
 *   sq, sk      sequence lengths (must equal tiles->sq, tiles->sk)
 *   hq, hk      query / key-value heads, hq % hk == 0 (grouped-query heads)
 *   d           head dim, 64 or 128
 *   scale       softmax scale (> 0, finite), applied to q . k
 *   tiles       metadata from attn_build_tiles with tile shape
 *               ATTN_FWD_TILE_Q x ATTN_FWD_TILE_K, or (d = 128 only)
 *               ATTN_FWD_PAIR_TILE_Q x ATTN_FWD_TILE_K for the CTA-pair
 *               kernel (clusters of two CTAs; the attn_set_exp2_poly mode
 *               does not apply to it: every exponential stays on MUFU)
 *   out         [sq, hq, d] of out_dtype (ATTN_DTYPE_BF16 or _F32)
 *   lse         [hq, sq] f32: ln sum exp(scale q.k) over valid keys
 * A query row with no valid key gets O = 0 and lse = -inf.  q, k and v must
 * not overlap out (INVALID_ARG).
 * Each launch takes one of 4096 library-owned work counters in turn (a
 * counter starts at 0 and the launch puts it back to 0 when it ends).  A
 * launch captured in a CUDA graph keeps the counter it took, so replays of
 * one captured launch must not run concurrently with each other, nor with
 * the launch that takes the same counter 4096 launches later; otherwise two
 * grids share one counter and rows come out wrong.
 * Errors: INVALID_ARG, UNSUPPORTED (d, tile shape, misaligned pointer), CUDA.
 * Errors found on the device are reported by attn_last_device_error(): a
 * stalled pipeline stage gives up after a bounded wait (TIMEOUT), and
 * metadata whose build did not finish with ATTN_OK is not read at all (its
 * status); the outputs are then incomplete. */
int attn_fwd(const void *q, const void *k, const void *v, int sq, int sk, int hq, int hk, int d,
             float scale, const attn_tiles_t *tiles, void *out, int out_dtype, float *lse,
             attn_stream_t stream);

/* Exact merge of KV-split partials (UltraAttn page, section 3.2): with
 * m = max_i lse_i, w_i = exp(lse_i - m), L = sum_i w_i:
 *   lse = m + ln L,   O = sum_i (w_i / L) O_i.
 * Partials with lse_i = -inf drop out; if every partial is -inf, O = 0 and
 * lse = -inf.
 *   h_o_parts    host array of n_parts device pointers to [s_len, h, d] O_i
 *                of part_dtype (16-byte aligned)
 *   h_lse_parts  host array of n_parts device pointers to [h, s_len] f32
 *   n_parts      1..ATTN_MERGE_MAX_PARTS
 *   out, lse     [s_len, h, d] of out_dtype, [h, s_len] f32 (may not alias
 *                the inputs)
 * Errors: INVALID_ARG, UNSUPPORTED (d not in {64, 128}, alignment), CUDA. */
int attn_merge(const void *const *h_o_parts, const float *const *h_lse_parts, int n_parts,
               int part_dtype, int s_len, int h, int d, void *out, int out_dtype, float *lse,
               attn_stream_t stream);

/* Backward pass of the masked attention forward: gradients of a loss L with
 * respect to Q, K, V given dO = dL/dO, for the same tile metadata.  P is
 * recomputed from the forward's lse:  D = rowsum(dO * O),  dP = dO V^T,
 * dS = P * (dP - D),  dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K
 * (heads of a GQA group summed into dK, dV).  The pages list the backward
 * pass alongside the forward (MagiAttention page: forward and backward kernel
 * benchmarks; FlashAttention-4 page: a rebuilt backward pipeline); the
 * formulas are the chain rule through the softmax.
 *   q, k, v, dout   bf16 [S_q,H,d], [S_k,H_k,d], [S_k,H_k,d], [S_q,H,d]
 *   out, out_dtype  the forward output O (bf16 or f32) for D
 *   lse             [H, S_q] f32 from the forward
 *   dq, dk, dv      [S_q,H,d], [S_k,H_k,d], [S_k,H_k,d] of grad_dtype
 *   d_ws            >= attn_bwd_workspace_bytes() bytes (D, transposed lists)
 * No atomics: dK, dV are accumulated per key tile over its query tiles (a
 * transposed copy of the lists built on the device), dQ per query tile.
 * Errors: as attn_fwd (including the refusal of metadata whose status is not
 * ATTN_OK), plus CAPACITY when ws_bytes is too small. */
int attn_bwd_workspace_bytes(const attn_tiles_t *tiles, int hq, size_t *bytes);
int attn_bwd(const void *q, const void *k, const void *v, const void *out, int out_dtype,
             const void *dout, const float *lse, int sq, int sk, int hq, int hk, int d, float scale,
             const attn_tiles_t *tiles, void *dq, void *dk, void *dv, int grad_dtype, void *d_ws,
             size_t ws_bytes, attn_stream_t stream);

/* Synchronises `stream`, then returns and clears the device-side failure
 * status of the metadata build, forward and backward kernels on the current
 * device: ATTN_OK, ATTN_ERR_TIMEOUT when a bounded wait ran out (a build's
 * grid barrier, a forward or backward pipeline stage), or the status of
 * refused metadata.  The first failure of each kernel family is kept.  The
 * status words are per device, not per stream: a caller that runs launches
 * on several streams cannot tell from here which launch failed, and should
 * synchronise all of them before reading. */
int attn_last_device_error(attn_stream_t stream);

/* Sets the bound on every device-side wait of later attn_fwd launches on the
 * current process (nanoseconds; default 4e9).  Used to test the timeout path
 * with a short limit. */
int attn_set_wait_limit_ns(int64_t ns);

/* Selects where the exponentials of later attn_fwd launches (this process)
 * run.  FlashAttention-4 page, first technique: part of the exponentials on
 * the FMA units through a polynomial approximation, the rest on the
 * special-function unit (MUFU), which that page notes runs twice as fast on
 * GB300 as on B200.
 *   period 0   every exponential on the special-function unit (default)
 *   period 4/8 on FULL tiles, every 4th / 8th pair of exponentials of a row
 *              through a cubic for 2^f after range reduction (worst relative
 *              error 1.2e-4, below the bf16 rounding of P); MASKED tiles
 *              always use the special-function unit
 * Any other period: ATTN_ERR_INVALID_ARG.  Results stay within the forward's
 * tolerances either way; the mode only trades special-function work for
 * FMA-pipe instructions. */
int attn_set_exp2_poly(int period);

/* Failure-path self test: launches one CTA that waits, with the current wait
 * bound, on a barrier nothing will ever complete; the wait gives up, records
 * ATTN_ERR_TIMEOUT in the device status and the kernel returns normally.  Read
 * the result with attn_last_device_error(). */
int attn_selftest_wait_timeout(attn_stream_t stream);

/* Human-readable text of a status code (static storage). */
const char *attn_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* ATTN_SLICE_H */
