/*
 * attn_block_mask.h - C ABI of the GB300 (sm_103a) structured-mask attention
 * forward: a block-mask builder and the attention forward that consumes it.
 *
 * What is computed
 *   For every packed sequence b (tokens cu_seqlens[b] .. cu_seqlens[b+1]-1),
 *   every head h and every query token i of that sequence:
 *       O[i,h,:]  = sum_j softmax_j(scale * q_i . k_j) v_j   over visible j
 *       LSE[h,i]  = ln sum_j exp(scale * q_i . k_j)           over visible j
 *   where "visible" is the mask predicate of the chosen kind evaluated on the
 *   global packed token indices i, j of the same sequence ("Triton from first
 *   principles" Ch. 21, Sections 21.1-21.2: online-softmax flash attention with
 *   causal masking inside the loop).  Keys of other sequences are never
 *   visible (cu_seqlens packing, xorl issue "Block-mask attention:
 *   shared-prefix and strip-thinking", Summary).
 *
 * Mask kinds (predicates on global token indices qi, ki of one sequence)
 *   ATTN_MASK_CAUSAL           ki <= qi (diagonal included; Ch. 9, Section 9.1)
 *   ATTN_MASK_CAUSAL_DOCUMENT  ki <= qi and seg_id[ki] == seg_id[qi]
 *                              (xorl issue, Decisions, item 4: document
 *                              boundaries inside the mask)
 *   ATTN_MASK_SHARED_PREFIX    (qi >= ki) & ((seg[ki] == 0) | (seg[ki] == seg[qi]))
 *                              (xorl issue, Mask specifications, "Shared prefix")
 *   ATTN_MASK_STRIP_THINKING   (qi >= ki) & ~((role[ki] == THINK) & (turn[ki] < turn[qi]))
 *                              (xorl issue, Mask specifications, "Strip-thinking")
 *   ATTN_MASK_STRIP_THINKING_DUP  the exact variant with every answer span
 *                              duplicated (xorl issue, "The exactness
 *                              question", option (b)).  Roles: THINK =
 *                              role_think, ANSWER = 2 (the copy that sees its
 *                              own turn's thinking), ANSWER_HISTORY = 3 (the
 *                              copy later turns see), anything else context.
 *                              With ki <= qi, a key is visible when it is
 *                              context; THINK of the query's turn and the query
 *                              THINK or ANSWER; ANSWER of the query's turn and
 *                              the query ANSWER; ANSWER_HISTORY of an earlier
 *                              turn, or of the query's turn with the query
 *                              ANSWER_HISTORY.  role_think must not be 2 or 3.
 *   ATTN_MASK_NONE             every key of the sequence (no mask inside a
 *                              sequence; "Triton from first principles"
 *                              Ch. 21, Section 21.1, the plain kernel)
 *   ATTN_MASK_DENSE            the caller's bits (attn_mask_params.dense_bits):
 *                              any pattern, e.g. causal + document + padding
 *                              composed by the caller (xorl issue, "Current
 *                              state in this tree", make_causal_block_mask).
 *                              Sequence b's rows are L = cu[b+1] - cu[b] rows
 *                              of ceil(L / 32) uint32 words starting at word
 *                              dense_offsets[b]; key j of row i is bit j % 32
 *                              of word j / 32 of row i, 1 = visible; bits past
 *                              a row's end are ignored.
 * Rows that see no key get O = 0 and LSE = -inf (possible only for DENSE).
 *
 * Tiles
 *   Each sequence is cut into 128-token tiles starting at its first token.
 *   A (q-tile, k-tile) pair of one sequence is EMPTY when no in-bounds pair is
 *   visible, FULL when all are, PARTIAL otherwise ("Triton from first
 *   principles" Ch. 21, Section 21.2 diagram: all-valid / diagonal / skipped).
 *   EMPTY pairs are never loaded (Ch. 9, Section 9.2: skip whole tiles on a
 *   scalar flag); the predicate is evaluated only on PARTIAL pairs and the
 *   bounds test only on a sequence's ragged last tile.
 *
 * Conventions
 *   - Every array argument is a DEVICE pointer owned by the caller unless the
 *     comment says otherwise.  The library allocates no device memory.
 *   - The persistent kernels take their work counters from a small pool held
 *     by the library on each device (256 slots per kernel family, handed out
 *     round robin, each returned to zero by its launch's last CTA).  Up to
 *     256 forward and 256 backward launches may therefore be in flight on a
 *     device at once, on any streams; more than that could share a slot.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and return after host-side argument checks; a returned
 *     error means nothing was launched.
 *   - Errors found on the device (malformed cu_seqlens, a sequence longer
 *     than max_seqlen, a pipeline wait that timed out) are recorded in an
 *     error word inside the block-mask workspace and reported by
 *     attn_get_status().  No kernel traps or aborts.
 *   - Layouts: q, k, v, o are [total_tokens, num_heads, head_dim] row-major,
 *     contiguous, 16-byte aligned; lse is fp32 [num_heads, total_tokens].
 */
#ifndef ATTN_BLOCK_MASK_H
#define ATTN_BLOCK_MASK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* attn_stream_t;

typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,          /* NULL pointer, bad size, misaligned buffer */
  ATTN_ERR_UNSUPPORTED = 2,          /* valid but not implemented (e.g. head_dim 96) */
  ATTN_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below attn_block_mask_workspace_size() */
  ATTN_ERR_MASK_MISMATCH = 4,        /* block mask built for another kind / cu_seqlens / sizes */
  ATTN_ERR_CUDA = 5,                 /* a CUDA runtime or driver call failed */
  ATTN_ERR_DEVICE_TIMEOUT = 6,       /* a kernel gave up on a pipeline wait (reported later) */
  ATTN_ERR_DEVICE_INVALID_INPUT = 7  /* the device found cu_seqlens malformed (reported later) */
} attn_status;

typedef enum attn_mask_kind {
  ATTN_MASK_CAUSAL = 0,
  ATTN_MASK_CAUSAL_DOCUMENT = 1,
  ATTN_MASK_SHARED_PREFIX = 2,
  ATTN_MASK_STRIP_THINKING = 3,
  ATTN_MASK_STRIP_THINKING_DUP = 4,
  ATTN_MASK_NONE = 5,
  ATTN_MASK_DENSE = 6
} attn_mask_kind;

typedef enum attn_dtype {
  ATTN_DTYPE_BF16 = 0, /* bf16 in and out, fp32 accumulation (tcgen05 tensor cores) */
  ATTN_DTYPE_FP32 = 1  /* fp32 in and out, fp32 arithmetic (CUDA cores) */
} attn_dtype;

/* Tile labels stored in the block mask. */
#define ATTN_TILE_EMPTY 0
#define ATTN_TILE_PARTIAL 1
#define ATTN_TILE_FULL 2

/* Tile size of the block mask (rows x columns of one (q-tile, k-tile) pair). */
#define ATTN_BLOCK_M 128
#define ATTN_BLOCK_N 128

typedef struct attn_mask_params {
  int32_t role_think; /* role code of THINK tokens for the STRIP_THINKING kinds (default 1) */
  const uint32_t* dense_bits;    /* device, ATTN_MASK_DENSE only: the bit rows */
  const int64_t* dense_offsets;  /* device int64[batch + 1], ATTN_MASK_DENSE only: first
                                    word of each sequence's rows */
} attn_mask_params;

/*
 * Block mask: a plain struct filled by attn_block_mask_build(), owned by the
 * caller, describing arrays that live in the caller's device workspace.
 * Byte offsets (off_*) are from the workspace base; array sizes are in the
 * comments, with NQ = max_qtiles and NK = max_ktiles.
 *   off_header  int32[16]: [0] n_qtiles, [1] n_entries (sum of kcount),
 *               [2] error bits, [3] n_qpairs, [4] EMPTY, [5] PARTIAL,
 *               [6] FULL tile-pair totals, others reserved.  The kernels
 *               only read the mask (their work counters belong to each
 *               launch), so attn_fwd and attn_bwd calls that share one block
 *               mask may run concurrently on different streams, as long as
 *               no attn_block_mask_build rewrites the workspace meanwhile.
 *   off_qt_seq  int32[NQ]       sequence of each q-tile (q-tiles are numbered
 *                               sequence-major, ascending inside a sequence)
 *   off_qt_idx  int32[NQ]       index of the q-tile inside its sequence
 *   off_labels  uint8[NQ * NK]  row g = labels of q-tile g against k-tiles
 *                               0 .. n_ktiles(seq)-1 of its own sequence
 *   off_kcount  int32[NQ]       number of non-EMPTY k-tiles of each q-tile
 *   off_koff    int32[NQ + 1]   CSR offsets into kidx / klabel
 *   off_kidx    int32[NQ * NK]  ascending k-tile indices (inside the sequence)
 *   off_klabel  uint8[NQ * NK]  ATTN_TILE_PARTIAL or ATTN_TILE_FULL per entry
 *   off_order   int32[NQ]       q-tiles by descending kcount, ties by index
 *   off_qt_off  int32[batch+1]  first q-tile number of each sequence
 *   off_summary int32[NQ * 8]   per-tile metadata summary used by the classifier
 *   off_pair_off   int32[batch+1]  first q-tile-pair number of each sequence
 *   off_pair_q0    int32[NQ]       first q-tile of each q-tile pair; a pair is
 *                                  q-tiles (2j, 2j+1) of one sequence, the second
 *                                  absent when the sequence has an odd count
 *   off_pair_order int32[NQ]       q-tile pairs by descending summed kcount,
 *                                  ties by pair number
 * The transposed (k-major) lists the backward walks: k-tiles are numbered like
 * q-tiles (tile g of its sequence is k-tile g, for the same g), and
 *   off_qcount  int32[NQ]       number of non-EMPTY q-tiles of each k-tile
 *   off_qoff    int32[NQ + 1]   CSR offsets into qidx / qlabel
 *   off_qidx    int32[NQ * NK]  ascending q-tile indices (inside the sequence)
 *   off_qlabel  uint8[NQ * NK]  ATTN_TILE_PARTIAL or ATTN_TILE_FULL per entry
 *   off_korder  int32[NQ]       k-tiles by descending qcount, ties by index
 */
typedef struct attn_block_mask {
  uint32_t magic;          /* set by the builder; checked by attn_fwd */
  int32_t kind;            /* attn_mask_kind */
  int32_t role_think;
  int32_t batch;
  int32_t total_tokens;
  int32_t max_seqlen;
  int32_t block_m;
  int32_t block_n;
  int32_t max_qtiles;      /* NQ = ceil(total_tokens / block_m) + batch */
  int32_t max_ktiles;      /* NK = ceil(max_seqlen / block_n) */
  const int32_t* cu_seqlens; /* device pointer the mask was built from */
  const uint32_t* dense_bits;    /* ATTN_MASK_DENSE: the params it was built from */
  const int64_t* dense_offsets;
  void* workspace;
  size_t workspace_bytes;
  uint64_t off_header, off_qt_seq, off_qt_idx, off_labels, off_kcount, off_koff,
      off_kidx, off_klabel, off_order, off_qt_off, off_summary, off_pair_off, off_pair_q0,
      off_pair_order, off_qcount, off_qoff, off_qidx, off_qlabel, off_korder;
} attn_block_mask;

/*
 * Bytes of device workspace attn_block_mask_build() needs for these sizes.
 * block_m and block_n must both be 128 (the tcgen05 M=128 tile).  Pure host
 * function: no CUDA call.  Returns ATTN_ERR_INVALID_ARG for negative sizes,
 * bytes == NULL or an overflow, ATTN_ERR_UNSUPPORTED for other tile sizes.
 */
ATTN_API attn_status attn_block_mask_workspace_size(int32_t batch, int32_t total_tokens,
                                           int32_t max_seqlen, int32_t block_m,
                                           int32_t block_n, size_t* bytes);

/*
 * Build the block mask of `kind` for the packed batch described by
 * cu_seqlens (device int32[batch+1], cu_seqlens[0] = 0, non-decreasing,
 * cu_seqlens[batch] = total_tokens, every length <= max_seqlen) and the
 * per-token metadata the kind needs (device arrays of total_tokens entries):
 *   CAUSAL: none; CAUSAL_DOCUMENT and SHARED_PREFIX: seg_id;
 *   STRIP_THINKING and STRIP_THINKING_DUP: role and turn; NONE: none; DENSE:
 *   params->dense_bits and params->dense_offsets.  Unused pointers may be
 *   NULL.
 * The mask is built once and can be reused by any number of attn_fwd calls
 * while the metadata does not change (xorl issue, Proposed work, item 3:
 * masks compiled and cached across steps).  It follows the forward (q-major)
 * orientation: per q-tile lists of k-tiles.
 * Labels are exact: whenever the per-tile metadata summaries cannot decide a
 * tile pair, the builder counts the predicate over the pair's tokens.
 * params may be NULL (role_think = 1).  `out` (host) receives the
 * description; workspace (device, >= attn_block_mask_workspace_size bytes,
 * 256-byte aligned) holds the arrays and must outlive every use of `out`.
 * Malformed cu_seqlens is detected on the device: the mask then has no
 * q-tiles and attn_get_status() returns ATTN_ERR_DEVICE_INVALID_INPUT.
 */
ATTN_API attn_status attn_block_mask_build(attn_mask_kind kind, const attn_mask_params* params,
                                  const int32_t* cu_seqlens, int32_t batch,
                                  int32_t total_tokens, int32_t max_seqlen,
                                  const int32_t* seg_id, const int8_t* role,
                                  const int32_t* turn, int32_t block_m, int32_t block_n,
                                  void* workspace, size_t workspace_bytes,
                                  attn_block_mask* out, attn_stream_t stream);

/*
 * Attention forward with the structured mask (see the top of this file).
 *   q, k, v   device [total_tokens, num_heads, head_dim], dtype `dtype`
 *   o         device output, same layout and dtype (rows of every sequence
 *             are written; nothing else is touched)
 *   lse       device fp32 [num_heads, total_tokens] output (natural log)
 *   head_dim  32, 64 or 128
 *   scale     score scale; 0 means 1/sqrt(head_dim)
 *   cu_seqlens, batch, max_seqlen, kind, params, seg_id, role, turn: the same
 *             values the block mask was built from (checked: kind, the
 *             cu_seqlens pointer, batch, total_tokens, max_seqlen, role_think,
 *             and for DENSE the two dense pointers)
 *   bm        the block mask from attn_block_mask_build()
 * bf16 runs on the tensor cores (tcgen05, fp32 accumulation in tensor
 * memory, P rounded to bf16 for the P.V product, O rounded to nearest even);
 * fp32 runs on the CUDA cores in fp32.  Deterministic: no atomics on the
 * output and a fixed k-tile order, so repeated calls are bit-identical.
 */
ATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     attn_dtype dtype, int32_t total_tokens, int32_t num_heads,
                     int32_t head_dim, float scale, const int32_t* cu_seqlens,
                     int32_t batch, int32_t max_seqlen, attn_mask_kind kind,
                     const attn_mask_params* params, const int32_t* seg_id,
                     const int8_t* role, const int32_t* turn, const attn_block_mask* bm,
                     attn_stream_t stream);

/*
 * Bytes of device workspace attn_bwd() needs for `num_heads` heads of
 * `head_dim` (32, 64 or 128) over the mask `bm` (built by
 * attn_block_mask_build()).  Pure host function.  The workspace holds,
 * 256-byte aligned:
 *   D = rowsum(dout * o)        fp32 [num_heads, total_tokens]
 *   ||dout_i||                  fp32 [num_heads, total_tokens]
 *   bound words                 fp32 [batch][num_heads][4]: the largest
 *                               ||v_j|| and |k_jd| of each sequence and
 *                               head (word 2 of the first: the call's
 *                               work-order head-group size, int32; the
 *                               other spare words unused)
 *   dQ accumulator              int32 [total_tokens, num_heads, head_dim],
 *                               fixed point
 * i.e. O(total_tokens * num_heads * head_dim); nothing is kept per tile pair.
 * Returns ATTN_ERR_UNSUPPORTED for another head_dim.
 */
ATTN_API attn_status attn_bwd_workspace_size(const attn_block_mask* bm, int32_t num_heads,
                                             int32_t head_dim, size_t* bytes);

/*
 * Attention backward with the structured mask: the gradients of attn_fwd()'s
 * O with respect to q, k and v for an upstream gradient dout ("the xorl issue",
 * Verified FA4 gaps, items 1-3: a backward over the same block-sparse masks,
 * walking the transposed lists for dK and dV, with a deterministic dQ).
 *   q, k, v, o, dout  device bf16 [total_tokens, num_heads, head_dim]: the
 *             forward's inputs, its output O and dL/dO
 *   lse       device fp32 [num_heads, total_tokens]: the forward's LSE
 *   dq, dk, dv  device bf16 outputs, layout of q (rows of every sequence are
 *             written; nothing else is touched)
 *   head_dim, scale, cu_seqlens, batch, max_seqlen, kind, params, seg_id,
 *             role, turn, bm: as for attn_fwd(), with the same checks; the
 *             block mask's transposed (k-major) lists drive the work
 *   workspace device, 256-byte aligned, caller-owned scratch of at least
 *             attn_bwd_workspace_size() bytes (layout above), else
 *             ATTN_ERR_WORKSPACE_TOO_SMALL
 * Math: P = exp(scale q k^T - LSE) over the visible pairs, dV = P^T dO,
 * dP = dO V^T, dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q.  One
 * persistent kernel walks every (k-tile, head)'s list: five tensor-core
 * products per visible tile pair (S^T, dP^T, dV, dK and dQ^T = K^T dS^T), with
 * dS kept on chip.  Each k-tile's dQ^T contribution is added into an int32
 * fixed-point accumulator whose quantum, per query row i and head, is 2^-30
 * of 4 ||dout_i|| max_j||v_j|| max_jd|k_jd| (the maxima over the row's
 * sequence; twice a bound on every partial sum of the row, so the sums never
 * overflow); integer addition is exact, so the backward is deterministic
 * (bit-identical repeats, whatever the order of the adds) without per-pair
 * storage.  P and dS are rounded to bf16 for the
 * tensor-core products, accumulation is fp32 in tensor memory, outputs are
 * rounded to nearest even.  `lse` must be the forward's (the bound assumes
 * each row's weights sum to one).  Inputs must be finite inside each
 * sequence.  Only ATTN_DTYPE_BF16 exists
 * (ATTN_ERR_UNSUPPORTED otherwise).  Launches that share one block mask may
 * run concurrently with each other and with attn_fwd() on other streams, each
 * with its own workspace.
 */
ATTN_API attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              attn_dtype dtype, int32_t total_tokens, int32_t num_heads,
                              int32_t head_dim, float scale, const int32_t* cu_seqlens,
                              int32_t batch, int32_t max_seqlen, attn_mask_kind kind,
                              const attn_mask_params* params, const int32_t* seg_id,
                              const int8_t* role, const int32_t* turn,
                              const attn_block_mask* bm, void* workspace, size_t workspace_bytes,
                              attn_stream_t stream);

/*
 * Same as attn_block_mask_build(), for callers that cannot allocate device
 * memory (a host memory manager that owns every device byte, or a loop where
 * an allocation and its implicit synchronisation are not allowed).  The pages
 * have no counterpart: this is a deployment variant of the builder.
 *   - Same arguments and the same output: the block-mask arrays attn_fwd()
 *     reads (header, q-tile descriptors, kcount, koff, kidx, klabel, order,
 *     q-tile pairs) are written to `workspace` at the usual offsets
 *     (workspace_bytes >= attn_block_mask_workspace_size()).
 *   - The builder's temporary arrays (tile summaries, the dense tile-label
 *     matrix, per-sequence offsets) live in a fixed 4 MiB device array inside
 *     the library instead; they are not kept, so off_labels, off_summary,
 *     off_qt_off and off_pair_off name unwritten workspace regions.
 *   - Needs max_qtiles * max_ktiles + 32 * max_qtiles + 8 * (batch + 1) bytes
 *     of that array (each part rounded up to 256): up to 259,968 tokens in one
 *     sequence; larger problems return ATTN_ERR_UNSUPPORTED and launch
 *     nothing.
 *   - The first call on a device looks up the array's address with that device
 *     current; make that first call before any stream capture.  The address is
 *     kept for the life of the process, so after cudaDeviceReset (which makes a
 *     new context) this entry point must not be called on that device again.
 *   - All calls on a device share the array: calls whose kernels overlap on the
 *     GPU race and must be serialised by the caller.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
ATTN_API attn_status attn_block_mask_build_noalloc(
    attn_mask_kind kind, const attn_mask_params* params, const int32_t* cu_seqlens, int32_t batch,
    int32_t total_tokens, int32_t max_seqlen, const int32_t* seg_id, const int8_t* role,
    const int32_t* turn, int32_t block_m, int32_t block_n, void* workspace, size_t workspace_bytes,
    attn_block_mask* out, attn_stream_t stream);

/*
 * Synchronise `stream`, then report the device error word of `bm` (and any
 * pending CUDA error): ATTN_OK, ATTN_ERR_DEVICE_INVALID_INPUT,
 * ATTN_ERR_DEVICE_TIMEOUT or ATTN_ERR_CUDA.  The error word is cleared by the
 * next attn_block_mask_build() on the same workspace.
 */
ATTN_API attn_status attn_get_status(const attn_block_mask* bm, attn_stream_t stream);

/*
 * The CUDA runtime's message for the last CUDA failure this library saw on the
 * calling thread (the one behind the most recent ATTN_ERR_CUDA), or "" if none.
 * The string is owned by the library and stays valid until the next call on
 * this thread.
 */
ATTN_API const char* attn_last_error_message(void);

/* Static, NUL-terminated description of a status code. */
ATTN_API const char* attn_status_string(attn_status status);

/* Library version as an integer (major * 10000 + minor * 100 + patch). */
ATTN_API int32_t attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BLOCK_MASK_H */
