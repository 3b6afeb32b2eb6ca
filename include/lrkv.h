/*
 * lrkv.h - C ABI of the GB300 (sm_103a) LRKV decode / append / prefill library.
 *
 * Low-Rank Key Value attention (LRKV) caches, per layer and token, one shared
 * key row S_K and one shared value row S_V (width d_h) plus, per head h, a
 * private key row R_K[h] and value row R_V[h] (width r).  A head's key is
 * S_K + R_K[h] B_K[h]^T and its value S_V + R_V[h] B_V[h]^T, where B_K[h],
 * B_V[h] (d_h x r) are layer weights (reading note "Low-Rank Key Value
 * Attention", section 3, equations 2-5).  Decode never materialises those
 * keys or values: it scores q.S_K + (q B_K[h]).R_K[h] (equation 6) and reduces
 * values as a.S_V + (a.R_V[h]) B_V[h]^T (equation 7), with one softmax over
 * both score branches and scale 1/sqrt(d_h) (section 2).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All tensor pointers are DEVICE pointers, 16-byte aligned, row-major and
 *    dense.  The library only reads inputs, writes only the listed outputs and
 *    the addressed cache slots, never frees or keeps any pointer past the call,
 *    and allocates nothing.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *    A return of LRKV_OK means the work was validated and enqueued.
 *  - Element type: every floating tensor of one call (X, Q, q, weights, bases,
 *    cache pools, out) has the cache's dtype (LRKV_F32 or LRKV_BF16).  All
 *    arithmetic accumulates in fp32; results are rounded once on store.
 *  - Errors the host can see (null pointers, bad sizes, too-small workspace,
 *    unsupported dtype) are returned as a negative LRKV_E_* code before any
 *    work is enqueued.  Errors in device-resident metadata (a page id outside
 *    [0, num_pages), a sequence length outside [1, max_pages*page_size], a
 *    position or sequence id out of range) are never turned into an access:
 *    the affected rows are skipped and the kernel ORs an LRKV_STATUS_* bit
 *    into *dev_status (a caller-owned device int32, may be NULL; the library
 *    never clears it).
 */
#ifndef LRKV_H
#define LRKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define LRKV_API __attribute__((visibility("default")))
#else
#define LRKV_API
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *lrkv_stream_t;

/*
 * Element types.  LRKV_F32 and LRKV_BF16 apply to every floating tensor of a
 * call.  LRKV_FP8_E4M3 stores the four cache pools as 8-bit E4M3 codes (OCP
 * 8-bit floating point: sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities, largest finite 448), each pool with its own scale
 * (lrkv_cache_t.scale); every other floating tensor of the call (X, weights,
 * q, Q, B_K, B_V, out) is bf16.  It halves the cache payload of equation 9.
 */
typedef enum { LRKV_F32 = 0, LRKV_BF16 = 1, LRKV_FP8_E4M3 = 2 } lrkv_dtype_t;

enum {
    LRKV_OK = 0,
    LRKV_E_INVALID_ARG = -1, /* null pointer, negative count, misaligned pointer */
    LRKV_E_SHAPE = -2,       /* a dimension is zero, too large or inconsistent */
    LRKV_E_DTYPE = -3,       /* dtype not an lrkv_dtype_t, or a scale not positive finite */
    LRKV_E_BOUNDS = -4,      /* host-visible bound: max_seq_len > max_pages*page_size, ... */
    LRKV_E_WORKSPACE = -5,   /* workspace NULL, misaligned or smaller than required */
    LRKV_E_CUDA = -6         /* a CUDA call failed; lrkv_last_cuda_error() has the code */
};

/* Bits ORed into *dev_status by the kernels. */
#define LRKV_STATUS_BAD_PAGE 1u     /* page id outside [0, num_pages) */
#define LRKV_STATUS_BAD_SEQLEN 2u   /* sequence length < 1 or > max_pages*page_size */
#define LRKV_STATUS_BAD_ROW 4u      /* append: position/sequence id out of range */
#define LRKV_STATUS_TIMEOUT 8u      /* an on-chip wait gave up (never expected) */

/*
 * Paged factored cache (section 3, after Algorithm 1: shared and private
 * pages use one token numbering and one lifetime).  Token t of request b
 * lives in page page_table[b*max_pages + t/page_size], slot t%page_size, and
 * that one page id indexes all four pools:
 *     S_K, S_V : [num_pages, page_size, d_h]
 *     R_K, R_V : [num_pages, page_size, H, r]   (all heads of a token contiguous)
 * Memory is caller-owned; the library never frees it.
 * Supported: 1 <= H <= 128, 1 <= d_h <= 256, 1 <= r <= 256, page_size a
 * multiple of 16 in [16, 1024]; with LRKV_BF16, d_h and r multiples of 8;
 * with LRKV_F32, multiples of 4; with LRKV_FP8_E4M3, d_h a multiple of 16, r
 * of 8 and H*r of 16.
 * With LRKV_FP8_E4M3 a pool with scale s stores, for a value x, the code of
 * x / s rounded to the nearest E4M3 value (ties to even, finite values beyond
 * +-448 saturating), and reads back decode(code) * s; scale[] is ignored for
 * the other dtypes.
 *
 * Joint key RMSNorm (reading note, section 8): when N_K is not NULL the cache
 * also holds, per token and head, the reciprocal root mean square of the full
 * key,  1 / sqrt(mean_d (S_K[j] + R_K[h,j] B_K[h]^T)_d^2 + norm_eps),
 *     N_K : [num_pages, page_size, H]   (bf16 for LRKV_BF16 and
 *            LRKV_FP8_E4M3 caches, fp32 for LRKV_F32; 16-byte aligned)
 * and every score is multiplied by it: s_j = (q.S_K[j] + p.R_K[h,j]) N_K[j,h]
 * / sqrt(d_h).  The values N_K holds are written by lrkv_key_norms (and by
 * lrkv_prefill and lrkv_decode_step for the rows they append).  A
 * per-channel gain and the query's own normalisation belong to q.  Costs one
 * scalar per head and token, 1/(2 d_h) of a dense K/V cache.
 *
 * Grouped shared basis (reading note, section 3 after equations 2-5: a basis
 * per group of heads whose needs differ): with G > 1 the heads form G groups
 * of H/G consecutive heads, each with its own shared projection, and a token
 * caches G shared rows:
 *     S_K, S_V : [num_pages, page_size, G, d_h]   (group-major)
 * head h reads group h / (H/G):  K_h = S_K[.., h/(H/G), :] + R_K[h] B_K[h]^T.
 * The shared weights of lrkv_append / lrkv_prefill / lrkv_decode_step are
 * then W_S_K, W_S_V [G*d_h, d] (group-major rows).  G must divide H; 0 and 1
 * both mean one shared basis.  The tiled prefill and the tensor-core rotary
 * decode serve G = 1 (other G take the per-row and generic kernels); the
 * tensor-core decode covers G = 1 and G = 2.
 */
typedef struct {
    void *S_K;
    void *S_V;
    void *R_K;
    void *R_V;
    int32_t num_pages;
    int32_t page_size;
    int32_t H;
    int32_t d_h;
    int32_t r;
    int32_t dtype;  /* lrkv_dtype_t */
    float scale[4]; /* LRKV_FP8_E4M3: scale of S_K, S_V, R_K, R_V (positive, finite) */
    void *N_K;      /* NULL, or the reciprocal key norms [num_pages, page_size, H] */
    float norm_eps; /* N_K: eps of the root mean square (finite, >= 0) */
    int32_t G;      /* shared key/value groups (0 or 1: one shared basis) */
} lrkv_cache_t;

/*
 * lrkv_append - build or extend the factored cache (section 3, Algorithm 1).
 *
 * For each of the n new rows X[i] (request seq_ids[i], token position
 * positions[i]):
 *     S_K = X W_S_K,  S_V = X W_S_V,  R_K[h] = X U_K[h],  R_V[h] = X U_V[h]
 * are computed with fp32 accumulation and stored (rounded to the cache dtype)
 * at the row's slot.  B_K, B_V are not needed: they stay layer weights.
 *
 *   X          [n, d]
 *   positions  [n] int32, device; seq_ids [n] int32, device, in [0, B)
 *   W_S_K      [d_h, d]     weights stored output-major (like nn.Linear.weight):
 *   W_S_V      [d_h, d]       row c holds the input weights of output column c
 *   U_K        [H, r, d]
 *   U_V        [H, r, d]
 *   page_table [B, max_pages] int32, device
 * Rows whose (seq_id, position, page id) are out of range are skipped and
 * flag LRKV_STATUS_BAD_ROW / LRKV_STATUS_BAD_PAGE.  Two rows that address the
 * same slot race (the caller must not do that).  n == 0 is a no-op.
 */
LRKV_API int lrkv_append(const void *X, const int32_t *positions, const int32_t *seq_ids,
                int32_t n, int32_t d, const void *W_S_K, const void *W_S_V,
                const void *U_K, const void *U_V, const lrkv_cache_t *cache,
                const int32_t *page_table, int32_t B, int32_t max_pages,
                int32_t *dev_status, lrkv_stream_t stream);

/* Bytes of device workspace lrkv_decode needs for these sizes. */
LRKV_API size_t lrkv_decode_workspace_bytes(int32_t B, int32_t H, int32_t d_h, int32_t r,
                                   int32_t max_seq_len, int32_t dtype);

/*
 * lrkv_decode - one decode step read directly from the factored cache
 * (section 3, Algorithm 2, equations 6 and 7).
 *
 * For request b and head h, over the seq_lens[b] cached rows j (the current
 * token included: decode runs after its row was appended):
 *     p        = q[b,h] B_K[h]                          (once per step)
 *     s_j      = (q[b,h].S_K[j] + p.R_K[h,j]) / sqrt(d_h)
 *     a        = softmax_j(s)                            (one softmax, both branches)
 *     out[b,h] = a.S_V + (a.R_V[h]) B_V[h]^T
 * Query projection, head concatenation and the output projection stay with
 * the caller.
 *
 *   q        [B, H, d_h]         out [B, H, d_h]
 *   B_K, B_V [H, d_h, r]
 *   seq_lens [B] int32, device; page_table [B, max_pages] int32, device
 *   max_seq_len  host upper bound of seq_lens (sizes the launch and workspace);
 *                must be <= max_pages*page_size.
 *   workspace    >= lrkv_decode_workspace_bytes(B, H, d_h, r, max_seq_len, dtype)
 *                bytes of device memory, 256-byte aligned, caller-owned; its
 *                contents are scratch (partial softmax states) and need no
 *                initialisation.
 * A request with an invalid length gets out = 0 and LRKV_STATUS_BAD_SEQLEN.
 */
LRKV_API int lrkv_decode(const void *q, const lrkv_cache_t *cache, const void *B_K,
                const void *B_V, const int32_t *seq_lens, const int32_t *page_table,
                int32_t B, int32_t max_pages, int32_t max_seq_len, void *out,
                void *workspace, size_t workspace_bytes, int32_t *dev_status,
                lrkv_stream_t stream);

/*
 * lrkv_decode_noalloc - the same decode step as lrkv_decode, for callers that
 * cannot allocate device memory.  (Library plumbing: the paper has no
 * counterpart.)
 *
 * Some hosts own every byte of device memory: a serving engine that reserves
 * HBM up front for its own pool, or a plugin hook whose contract forbids
 * allocating.  There, cudaMalloc either fails or stalls the whole device in
 * the middle of a latency-critical step, so such a caller cannot provide the
 * workspace lrkv_decode asks for.  This entry point takes the same arguments
 * minus the workspace and keeps its scratch (launch plan, private queries,
 * per-segment softmax partials) in a device array built into the library:
 *   - the array is LRKV_NOALLOC_SCRATCH_BYTES (16 MiB) on every GPU where the
 *     library's device code is loaded, held until the process exits.  CUDA
 *     loads device code lazily by default, so the array's memory is committed
 *     by the first call on each device, not when the library is opened: make
 *     that first call before the host reserves the rest of device memory for
 *     its own pool, and before any stream capture;
 *   - sizes whose lrkv_decode_workspace_bytes(B, H, d_h, r, max_seq_len,
 *     dtype) exceeds that are rejected with LRKV_E_WORKSPACE before any work;
 *   - every call looks up the array's device address with its device current
 *     (after the first call on a device this is a table read), so the entry
 *     point stays valid after the device's primary context is reset;
 *   - every call on a device shares the one array and leaves its scratch
 *     behind; nothing in it needs clearing (each call writes every value before
 *     reading it), but two calls that can run at the same time on the GPU
 *     (different streams, or threads) race: the caller must serialise them.
 * It allocates nothing and calls no allocating routine.
 */
#define LRKV_NOALLOC_SCRATCH_BYTES (16u << 20)
LRKV_API int lrkv_decode_noalloc(const void *q, const lrkv_cache_t *cache, const void *B_K,
                                 const void *B_V, const int32_t *seq_lens,
                                 const int32_t *page_table, int32_t B, int32_t max_pages,
                                 int32_t max_seq_len, void *out, int32_t *dev_status,
                                 lrkv_stream_t stream);

/*
 * lrkv_decode_step - one decode step together with the append of its new
 * rows (section 3: Algorithm 1 for the new row, then Algorithm 2 with
 * equations 6 and 7).  Request b's new row X[b] is projected and written at
 * position seq_lens[b] - 1, exactly where lrkv_append would put it, and
 * request b is decoded over its seq_lens[b] rows, that new one included, as
 * lrkv_decode would:
 *
 *   X [B, d]   one new row per request      q, out [B, H, d_h]
 *   W_S_K, W_S_V, U_K, U_V as lrkv_append; B_K, B_V, page_table and
 *   max_seq_len as lrkv_decode; seq_lens [B] counts the new row.
 *   workspace >= lrkv_decode_step_workspace_bytes(B, H, d_h, r, max_seq_len,
 *                dtype) bytes, 256-byte aligned, caller-owned scratch.
 *
 * Same result as lrkv_append (positions seq_lens[b] - 1, sequence ids b)
 * followed by lrkv_decode, up to floating-point rounding order.  The append
 * kernel takes each row's place from seq_lens itself (and so do the key
 * norms of a cache that keeps them), and the decode's first kernel, whose
 * inputs are none of the append's, runs beside it instead of after it.
 * A request with an invalid length gets no new row, out = 0 and
 * LRKV_STATUS_BAD_SEQLEN (with LRKV_STATUS_BAD_ROW from the append); a new
 * row on an invalid page is neither written nor attended and is flagged
 * LRKV_STATUS_BAD_PAGE.
 */
LRKV_API size_t lrkv_decode_step_workspace_bytes(int32_t B, int32_t H, int32_t d_h, int32_t r,
                                                 int32_t max_seq_len, int32_t dtype);
LRKV_API int lrkv_decode_step(const void *X, int32_t d, const void *W_S_K, const void *W_S_V,
                              const void *U_K, const void *U_V, const void *q,
                              const lrkv_cache_t *cache, const void *B_K, const void *B_V,
                              const int32_t *seq_lens, const int32_t *page_table, int32_t B,
                              int32_t max_pages, int32_t max_seq_len, void *out, void *workspace,
                              size_t workspace_bytes, int32_t *dev_status, lrkv_stream_t stream);

/*
 * lrkv_decode_step_host - lrkv_decode_step (reading note "Low-Rank Key Value
 * Attention", section 3: Algorithm 1 for the new rows, Algorithm 2 with
 * equations 6 and 7 for the queries) with the step's per-token inputs
 * and its output in HOST memory: the new rows X, the queries q and the
 * lengths seq_lens are copied to the device, the step runs, and out is
 * copied back, all enqueued on `stream` by this one call (it does not
 * synchronise: read out_host after the stream has reached this point).
 * Weights, bases, the cache and the page table stay on the device.
 *
 *   X_host [B, d], q_host [B, H, d_h], out_host [B, H, d_h]: host memory,
 *     element type as lrkv_decode_step; seq_lens_host [B] int32, host.
 *     Page-locked buffers (cudaHostAlloc / cudaHostRegister) are read and
 *     written through their device-mapped addresses: one copy kernel stages
 *     the inputs and the decode's last kernel stores out; pageable buffers go
 *     through the copy engines (cudaMemcpyAsync, which may then block).
 *   workspace >= lrkv_decode_step_host_workspace_bytes(B, H, d_h, r, d,
 *                max_seq_len, dtype) bytes of device memory, 256-byte
 *                aligned: the step's workspace plus device copies of the
 *                inputs and the output.
 *
 * Errors as lrkv_decode_step, checked before anything is enqueued; a failed
 * copy returns LRKV_E_CUDA.
 */
LRKV_API size_t lrkv_decode_step_host_workspace_bytes(int32_t B, int32_t H, int32_t d_h,
                                                      int32_t r, int32_t d, int32_t max_seq_len,
                                                      int32_t dtype);
LRKV_API int lrkv_decode_step_host(const void *X_host, int32_t d, const void *W_S_K,
                                   const void *W_S_V, const void *U_K, const void *U_V,
                                   const void *q_host, const lrkv_cache_t *cache, const void *B_K,
                                   const void *B_V, const int32_t *seq_lens_host,
                                   const int32_t *page_table, int32_t B, int32_t max_pages,
                                   int32_t max_seq_len, void *out_host, void *workspace,
                                   size_t workspace_bytes, int32_t *dev_status,
                                   lrkv_stream_t stream);

/*
 * Decode-step graphs - lrkv_decode_step_host recorded once as a CUDA graph
 * (the three input copies, the step's kernels with their programmatic
 * dependencies, the output copy) and replayed per step with one launch, so
 * the host's per-step cost is one graph launch instead of eight enqueues.
 *
 * lrkv_step_graph_create takes the arguments of lrkv_decode_step_host and
 * checks them the same way; nothing runs.  The graph keeps every pointer and
 * size it was made with: each lrkv_step_graph_launch reads X_host, q_host and
 * seq_lens_host as they are when the copies run (refill them between steps;
 * every length stays within max_seq_len) and writes out_host, which the
 * caller reads after synchronising the stream.  The cache, weights, page
 * table and workspace must stay allocated while the graph exists.
 *
 * Returns LRKV_OK and sets *graph, or an error (then *graph = NULL).
 * lrkv_step_graph_destroy frees a graph (NULL is a no-op); synchronise the
 * streams it was launched on first.
 */
typedef struct lrkv_step_graph_s *lrkv_step_graph_t;
LRKV_API int lrkv_step_graph_create(lrkv_step_graph_t *graph, const void *X_host, int32_t d,
                                    const void *W_S_K, const void *W_S_V, const void *U_K,
                                    const void *U_V, const void *q_host, const lrkv_cache_t *cache,
                                    const void *B_K, const void *B_V, const int32_t *seq_lens_host,
                                    const int32_t *page_table, int32_t B, int32_t max_pages,
                                    int32_t max_seq_len, void *out_host, void *workspace,
                                    size_t workspace_bytes, int32_t *dev_status);
LRKV_API int lrkv_step_graph_launch(lrkv_step_graph_t graph, lrkv_stream_t stream);
LRKV_API void lrkv_step_graph_destroy(lrkv_step_graph_t graph);

/* Bytes of device workspace lrkv_prefill needs. */
LRKV_API size_t lrkv_prefill_workspace_bytes(int32_t B, int32_t n, int32_t H, int32_t d_h,
                                    int32_t r, int32_t max_ctx, int32_t dtype);

/*
 * lrkv_prefill - append a chunk of new rows, then run causal LRKV attention
 * for every new row (section 2: prefill builds the first cache; section 3:
 * Algorithm 1 then equations 6-7 applied to every query row).
 *
 * Request b owns rows cu_rows[b] .. cu_rows[b+1]-1 of X, Q and out, at token
 * positions start_pos[b], start_pos[b]+1, ...; rows 0..start_pos[b]-1 must
 * already be in the cache (earlier history).  Row i at position t attends to
 * every row of its request at positions <= t:
 *     out[i,h] = softmax_j((Q[i,h].S_K[j] + (Q[i,h] B_K[h]).R_K[h,j]) / sqrt(d_h))
 *                applied to  S_V[j] + R_V[h,j] B_V[h]^T
 *
 *   X   [n, d]    Q, out [n, H, d_h]
 *   cu_rows [B+1] int32, device (cu_rows[0] = 0, nondecreasing, cu_rows[B] = n)
 *   start_pos [B] int32, device
 *   max_ctx   host upper bound of start_pos[b] + rows of b (<= max_pages*page_size)
 *   weights as lrkv_append; B_K, B_V as lrkv_decode.
 *   workspace >= lrkv_prefill_workspace_bytes(...) bytes, 256-byte aligned.
 */
LRKV_API int lrkv_prefill(const void *X, const void *Q, const int32_t *cu_rows,
                 const int32_t *start_pos, int32_t B, int32_t n, int32_t max_ctx,
                 int32_t d, const void *W_S_K, const void *W_S_V, const void *U_K,
                 const void *U_V, const void *B_K, const void *B_V,
                 const lrkv_cache_t *cache, const int32_t *page_table,
                 int32_t max_pages, void *out, void *workspace,
                 size_t workspace_bytes, int32_t *dev_status, lrkv_stream_t stream);

/*
 * Which attention kernel lrkv_prefill runs for this cache (host-only query):
 *   LRKV_PREFILL_TILED   - 128-row query tiles on the tensor cores, keys in
 *                          tiles of 64; taken for bf16 caches with d_h = 128,
 *                          r a multiple of 8 up to 64 and page_size a
 *                          multiple of 64, when tensor maps can be encoded;
 *   LRKV_PREFILL_PER_ROW - every query row as a one-query decode (any shape).
 * Both compute the same function.  Returns a negative LRKV_E_* code for an
 * invalid descriptor.
 */
#define LRKV_PREFILL_PER_ROW 0
#define LRKV_PREFILL_TILED 1
LRKV_API int lrkv_prefill_kernel_kind(const lrkv_cache_t *cache);

/*
 * lrkv_key_norms - store the reciprocal joint norm of the keys of n cached
 * rows (reading note, section 8): for row i (request seq_ids[i], position
 * positions[i], as in lrkv_append) and every head h,
 *     N_K[row, h] = 1 / sqrt(mean_d (S_K[row] + R_K[row, h] B_K[h]^T)_d^2 + norm_eps)
 * from the values the cache holds (call it after lrkv_append).  cache->N_K
 * must not be NULL.  Rows out of range are skipped and flagged like
 * lrkv_append's.  B_K [H, d_h, r] in the activation dtype.
 */
LRKV_API int lrkv_key_norms(const int32_t *positions, const int32_t *seq_ids, int32_t n,
                            const void *B_K, const lrkv_cache_t *cache, const int32_t *page_table,
                            int32_t B, int32_t max_pages, int32_t *dev_status,
                            lrkv_stream_t stream);

/*
 * Exact rotary position embedding over the factored cache (reading note,
 * section 8).  The cache keeps the unrotated projections S_K, S_V, R_K, R_V of
 * lrkv_append.  With D_j the rotation that turns channel pairs (2c, 2c+1) of
 * a row vector by j * theta_c, theta_c = base^(-2c/d_h) (all d_h channels,
 * (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos)), head h's key at position j
 * is (S_K[j] + R_K[h,j] B_K[h]^T) D_j and the query at position i is q D_i, so
 *     s_j = (q D_{i-j}).S_K[j] + ((q D_{i-j}) B_K[h]).R_K[h,j]   (/ sqrt(d_h))
 * -- the note's exact route (q~_i D_j^T B_h) z_j^T, which keeps z_j unrotated
 * and pays d_h*r multiply-adds per key and head.  Values are not rotated.
 * Key j of a request sits at position j; the decode query at seq_lens[b]-1,
 * a prefill row at its own position.
 *
 * lrkv_rope_table fills a table of lrkv_rope_table_bytes(d_h, max_pos) bytes
 * of device memory (16-byte aligned, caller-owned) with, for position p <
 * max_pos and channel pair c < d_h/2, (cos, sin)(p * theta_c) computed in
 * double precision: first as float pairs [max_pos][d_h/2][2] (rounded once),
 * then, from byte offset max_pos * d_h * 4 rounded up to a multiple of 256,
 * as f16 pairs in the same order (rounded once from the double, to nearest
 * even).  base > 1 and finite, d_h even in [2, 256], 1 <= max_pos <= 2^24.
 * lrkv_rope_table_bytes returns 0 for other sizes.
 *
 * lrkv_decode_rope / lrkv_prefill_rope take the arguments of lrkv_decode /
 * lrkv_prefill plus that table and its max_pos, which must be >= max_seq_len
 * (decode) or max_ctx (prefill).  d_h must be even and r <= 64.  Any cache
 * dtype.  lrkv_prefill_rope's workspace is lrkv_prefill's; lrkv_decode_rope
 * needs lrkv_decode_rope_workspace_bytes (lrkv_decode's plus room for the
 * rotated operands and one fp32 score per visible row and head).  On bf16
 * caches with d_h = 128, the tensor-core decode shapes and no key norms, lrkv_decode_rope
 * takes the angle-addition route D_{i-j} = D_i D_j^T: per step it forms
 * q~ = q D_i and the d_h x r matrix W_h with (q D_{i-j}) B_K[h] = C_j W_h,
 * C_j the key's (cos, sin) row; a score kernel evaluates q~.(S_K[j] D_j) +
 * (C_j W_h).R_K[h,j] on the tensor cores (f16 C_j and W_h, the rotated
 * S_K[j] and q~ in bf16, fp32 sums) and the split kernel attends with those
 * scores.  There, a request longer than max_seq_len or than the table is
 * not attended (zero output, LRKV_STATUS_BAD_SEQLEN).
 */
LRKV_API size_t lrkv_rope_table_bytes(int32_t d_h, int32_t max_pos);
LRKV_API int lrkv_rope_table(double base, int32_t d_h, int32_t max_pos, void *table,
                             lrkv_stream_t stream);
LRKV_API size_t lrkv_decode_rope_workspace_bytes(int32_t B, int32_t H, int32_t d_h, int32_t r,
                                                 int32_t max_seq_len, int32_t dtype);
LRKV_API int lrkv_decode_rope(const void *q, const lrkv_cache_t *cache, const void *B_K,
                              const void *B_V, const int32_t *seq_lens, const int32_t *page_table,
                              int32_t B, int32_t max_pages, int32_t max_seq_len,
                              const void *rope_table, int32_t rope_max_pos, void *out,
                              void *workspace, size_t workspace_bytes, int32_t *dev_status,
                              lrkv_stream_t stream);
LRKV_API int lrkv_prefill_rope(const void *X, const void *Q, const int32_t *cu_rows,
                               const int32_t *start_pos, int32_t B, int32_t n, int32_t max_ctx,
                               int32_t d, const void *W_S_K, const void *W_S_V, const void *U_K,
                               const void *U_V, const void *B_K, const void *B_V,
                               const lrkv_cache_t *cache, const int32_t *page_table,
                               int32_t max_pages, const void *rope_table, int32_t rope_max_pos,
                               void *out, void *workspace, size_t workspace_bytes,
                               int32_t *dev_status, lrkv_stream_t stream);

/*
 * Cache payload in bytes for `tokens` cached positions of one layer:
 * tokens * 2 * (d_h + H*r) * sizeof(dtype)  (section 4, equation 9).
 * Returns 0 for invalid arguments.
 */
LRKV_API size_t lrkv_cache_bytes(int32_t H, int32_t d_h, int32_t r, int64_t tokens, int32_t dtype);
/* The same with G shared groups (section 4, equation 9 with G shared rows per
 * token; the grouped variant of section 3): tokens * 2 * (G*d_h + H*r) *
 * sizeof(dtype); 0 for a G that does not divide H. */
LRKV_API size_t lrkv_cache_bytes_grouped(int32_t H, int32_t d_h, int32_t r, int32_t G,
                                         int64_t tokens, int32_t dtype);

/* Human-readable name of an LRKV_E_* code. */
LRKV_API const char *lrkv_status_string(int status);

/* cudaError_t of the last failed CUDA call inside the library (0 if none). */
LRKV_API int lrkv_last_cuda_error(void);

/*
 * Instrumentation for benchmarks.  lrkv_profile_enable(1) creates pools of
 * CUDA events (once) and starts recording: every later call brackets its
 * dominant kernel with an event pair on the call's stream -- the
 * split-attention kernel of lrkv_decode / lrkv_prefill (LRKV_PROFILE_ATTENTION),
 * the projection kernel of lrkv_append / lrkv_prefill
 * (LRKV_PROFILE_PROJECTION) and the rotary score kernel of lrkv_decode_rope's
 * tensor-core path (LRKV_PROFILE_SCORES); at most 8192 pairs are kept of each.
 * lrkv_profile_read(which, ...) waits for that kind's last event, returns its
 * summed kernel time in milliseconds and the number of bracketed launches,
 * and clears that record.  Not for use inside CUDA-graph capture.
 * lrkv_profile_enable(0) stops recording.
 */
#define LRKV_PROFILE_ATTENTION 0
#define LRKV_PROFILE_PROJECTION 1
#define LRKV_PROFILE_SCORES 2
LRKV_API int lrkv_profile_enable(int on);
LRKV_API int lrkv_profile_read(int32_t which, double *total_ms, int32_t *launches);

/* Library version, major*10000 + minor*100 + patch. */
LRKV_API int lrkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LRKV_H */
