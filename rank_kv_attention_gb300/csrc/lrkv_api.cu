// C-ABI entry points of the LRKV library: argument validation on the host,
// workspace layout, and dispatch to the kernels.  Nothing here allocates.
#include <math.h>
#include <algorithm>
#include <cmath>
#include <string.h>
#include <mutex>
#include <vector>

#include "append_kernels.cuh"
#include "decode_kernels.cuh"

namespace lrkv {

static thread_local int g_last_cuda_error = 0;

static int cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return LRKV_E_CUDA;
}

// Event pairs bracketing the dominant kernel of each call (benchmark
// instrumentation), one pool per kind.
struct Profiler {
    static const int kCap = 8192;
    bool created = false;
    int n = 0;
    cudaEvent_t ev[2 * kCap];
};
static bool g_prof_on = false;
static Profiler g_prof[3];

static void prof_before(int kind, cudaStream_t s) {
    Profiler &p = g_prof[kind];
    if (g_prof_on && p.n < Profiler::kCap) cudaEventRecord(p.ev[2 * p.n], s);
}
static void prof_after(int kind, cudaStream_t s) {
    Profiler &p = g_prof[kind];
    if (g_prof_on && p.n < Profiler::kCap) {
        cudaEventRecord(p.ev[2 * p.n + 1], s);
        ++p.n;
    }
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 160;  // no device visible (sizing queries only): an upper bound
    }
    return n;
}

cudaError_t smem_limit_once(const void *kern, int bytes) {
    struct Key {
        const void *kern;
        int dev, bytes;
    };
    static std::mutex mu;
    static std::vector<Key> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const Key &k : done)
        if (k.kern == kern && k.dev == dev && k.bytes == bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.push_back({kern, dev, bytes});
    return e;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

// Bytes of one cache element (the pools); activations of an 8-bit cache are bf16.
static int elem_bytes(int dtype) { return dtype == LRKV_F32 ? 4 : dtype == LRKV_BF16 ? 2 : 1; }

static int check_dims(int H, int d_h, int r, int dtype) {
    if (dtype != LRKV_F32 && dtype != LRKV_BF16 && dtype != LRKV_FP8_E4M3) return LRKV_E_DTYPE;
    if (H < 1 || H > 128 || d_h < 1 || d_h > 256 || r < 1 || r > 256) return LRKV_E_SHAPE;
    if (dtype == LRKV_FP8_E4M3) {  // 16-byte rows of codes; bf16 activations
        if (d_h % 16 || r % 8 || (H * r) % 16) return LRKV_E_SHAPE;
        return LRKV_OK;
    }
    const int mult = dtype == LRKV_BF16 ? 8 : 4;
    if (d_h % mult || r % mult) return LRKV_E_SHAPE;
    return LRKV_OK;
}

static int check_cache(const lrkv_cache_t *c) {
    if (!c) return LRKV_E_INVALID_ARG;
    int st = check_dims(c->H, c->d_h, c->r, c->dtype);
    if (st) return st;
    if (!c->S_K || !c->S_V || !c->R_K || !c->R_V) return LRKV_E_INVALID_ARG;
    if (!aligned16(c->S_K) || !aligned16(c->S_V) || !aligned16(c->R_K) || !aligned16(c->R_V))
        return LRKV_E_INVALID_ARG;
    if (c->num_pages < 1 || c->page_size < 16 || c->page_size > 1024 || c->page_size % 16)
        return LRKV_E_SHAPE;
    if ((int64_t)c->num_pages * c->page_size > INT32_MAX / 2) return LRKV_E_SHAPE;
    if (c->G < 0 || c->G > c->H || c->H % cache_groups(*c)) return LRKV_E_SHAPE;
    if (c->N_K && (!aligned16(c->N_K) || !(c->norm_eps >= 0.f) || !std::isfinite(c->norm_eps)))
        return LRKV_E_INVALID_ARG;
    if (c->dtype == LRKV_FP8_E4M3)
        for (int k = 0; k < 4; ++k)
            if (!(c->scale[k] > 0.f) || !std::isfinite(c->scale[k]) || !std::isfinite(1.f / c->scale[k]))
                return LRKV_E_DTYPE;
    return LRKV_OK;
}

// Decode launch geometry.  The workspace always reserves slots for the larger
// of the two paths' grids so that its size does not depend on the path.
struct DecodeGeom {
    int G_fast, G_gen, G_ws;
};

static DecodeGeom decode_geom(int B, int max_seq_len) {
    const int sm = device_sm_count();
    const int64_t rows = (int64_t)B * max_seq_len;
    DecodeGeom g;
    g.G_fast = (int)std::max<int64_t>(1, std::min<int64_t>(sm, (rows + 63) / 64));
    g.G_gen = (int)std::max<int64_t>(1, std::min<int64_t>(2 * sm, (rows + 255) / 256));
    g.G_ws = std::max(g.G_fast, g.G_gen);
    return g;
}

static size_t decode_ws_bytes(int B, int H, int d_h, int r, int max_seq_len) {
    DecodeGeom g = decode_geom(B, max_seq_len);
    return decode_ws_layout(nullptr, B, H, d_h, r, g.G_ws).bytes;
}

static int run_decode(const DecodeArgs &a, void *workspace, size_t ws_bytes) {
    const auto &c = a.cache;
    DecodeGeom geo = decode_geom(a.B, a.max_seq_len);
    DecodeWs ws = decode_ws_layout(workspace, a.B, c.H, c.d_h, c.r, geo.G_ws);
    if (ws_bytes < ws.bytes) return LRKV_E_WORKSPACE;
    const bool rope_fast = a.rope_ws.wt != nullptr;
    const bool fast = rope_fast || (!a.rope && fast_decode_supported(c.H, c.d_h, c.r, c.page_size, c.dtype,
                                                                      cache_groups(c)));
    const int G = fast ? geo.G_fast : geo.G_gen;
    cudaError_t e;
    if (c.dtype != LRKV_F32) {  // bf16 activations (bf16 or 8-bit cache)
        e = launch_prologue<__nv_bfloat16>(a, ws, G, kPlanTileAlign, fast);
        if (e == cudaSuccess && rope_fast) {
            prof_before(LRKV_PROFILE_SCORES, a.stream);
            e = launch_rope_scores(a, ws);
            prof_after(LRKV_PROFILE_SCORES, a.stream);
        }
        if (e == cudaSuccess) {
            prof_before(LRKV_PROFILE_ATTENTION, a.stream);
            e = fast ? launch_split_fast(a, ws, G) : launch_split_generic<__nv_bfloat16>(a, ws, G);
            prof_after(LRKV_PROFILE_ATTENTION, a.stream);
        }
        // the tensor-core split kernel merges the requests itself; the generic
        // one leaves that to the combine kernel
        if (e == cudaSuccess && !fast) e = launch_combine<__nv_bfloat16>(a, ws, G);
    } else {
        e = launch_prologue<float>(a, ws, G, kPlanTileAlign, false);
        if (e == cudaSuccess) {
            prof_before(LRKV_PROFILE_ATTENTION, a.stream);
            e = launch_split_generic<float>(a, ws, G);
            prof_after(LRKV_PROFILE_ATTENTION, a.stream);
        }
        if (e == cudaSuccess) e = launch_combine<float>(a, ws, G);
    }
    return e == cudaSuccess ? LRKV_OK : cuda_fail(e);
}

template <typename T>
static AppendArgsT<T> make_append_args(const void *X, const int32_t *positions,
                                       const int32_t *seq_ids, int n, int d, const void *W_S_K,
                                       const void *W_S_V, const void *U_K, const void *U_V,
                                       const lrkv_cache_t *c, const int32_t *page_table, int B,
                                       int max_pages, int32_t *status, cudaStream_t s) {
    AppendArgsT<T> a;
    a.X = static_cast<const T *>(X);
    a.positions = positions;
    a.seq_ids = seq_ids;
    a.n = n;
    a.d = d;
    a.W_S_K = static_cast<const T *>(W_S_K);
    a.W_S_V = static_cast<const T *>(W_S_V);
    a.U_K = static_cast<const T *>(U_K);
    a.U_V = static_cast<const T *>(U_V);
    a.S_K = static_cast<T *>(c->S_K);
    a.S_V = static_cast<T *>(c->S_V);
    a.R_K = static_cast<T *>(c->R_K);
    a.R_V = static_cast<T *>(c->R_V);
    a.page_table = page_table;
    a.B = B;
    a.max_pages = max_pages;
    a.num_pages = c->num_pages;
    a.page_size = c->page_size;
    a.H = c->H;
    a.d_h = c->d_h * cache_groups(*c);  // width of a token's shared row (all groups)
    a.r = c->r;
    a.status = status;
    a.stream = s;
    if (c->dtype == LRKV_FP8_E4M3) {
        a.fp8 = true;
        void *pools[4] = {c->S_K, c->S_V, c->R_K, c->R_V};
        for (int k = 0; k < 4; ++k) {
            a.q8[k] = static_cast<uint8_t *>(pools[k]);
            a.inv_scale[k] = 1.f / c->scale[k];
        }
        a.S_K = a.S_V = a.R_K = a.R_V = nullptr;
    }
    return a;
}

static int check_append(const void *X, const int32_t *positions, const int32_t *seq_ids, int n,
                        int d, const void *W_S_K, const void *W_S_V, const void *U_K,
                        const void *U_V, const lrkv_cache_t *cache, const int32_t *page_table,
                        int B, int max_pages) {
    int st = check_cache(cache);
    if (st) return st;
    if (n < 0 || B < 1 || max_pages < 1) return LRKV_E_SHAPE;
    if (d < 1 || d > 65536 || d % (cache->dtype == LRKV_F32 ? 4 : 8)) return LRKV_E_SHAPE;
    if ((int64_t)max_pages * cache->page_size > INT32_MAX / 2) return LRKV_E_SHAPE;
    if (n == 0) return LRKV_OK;
    if (!X || !positions || !seq_ids || !W_S_K || !W_S_V || !U_K || !U_V || !page_table)
        return LRKV_E_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W_S_K) || !aligned16(W_S_V) || !aligned16(U_K) ||
        !aligned16(U_V))
        return LRKV_E_INVALID_ARG;
    return LRKV_OK;
}

static int run_append(const void *X, const int32_t *positions, const int32_t *seq_ids, int n,
                      int d, const void *W_S_K, const void *W_S_V, const void *U_K,
                      const void *U_V, const lrkv_cache_t *c, const int32_t *page_table, int B,
                      int max_pages, int32_t *status, cudaStream_t s,
                      const int32_t *step_lens = nullptr) {
    // step_lens: row i is request i's row at position step_lens[i] - 1
    // (positions and seq_ids unused)
    if (n == 0) return LRKV_OK;
    cudaError_t e;
    prof_before(LRKV_PROFILE_PROJECTION, s);
    if (c->dtype != LRKV_F32) {  // bf16 rows and weights (bf16 or 8-bit cache)
        auto a = make_append_args<__nv_bfloat16>(X, positions, seq_ids, n, d, W_S_K, W_S_V, U_K,
                                                 U_V, c, page_table, B, max_pages, status, s);
        a.step_lens = step_lens;
        a.step_max_len = max_pages * c->page_size;
        if (rows_mma_append_fits(a)) e = launch_append_rows_mma(a);
        else if (rows_append_fits(a)) e = launch_append_rows(a);
        else if (tc_append_supported(n, d, c->d_h, c->H, c->r)) e = launch_append_tc(a);
        else e = launch_append_generic(a);
    } else {
        auto a = make_append_args<float>(X, positions, seq_ids, n, d, W_S_K, W_S_V, U_K, U_V, c,
                                         page_table, B, max_pages, status, s);
        a.step_lens = step_lens;
        a.step_max_len = max_pages * c->page_size;
        e = rows_append_fits(a) ? launch_append_rows(a) : launch_append_generic(a);
    }
    prof_after(LRKV_PROFILE_PROJECTION, s);
    return e == cudaSuccess ? LRKV_OK : cuda_fail(e);
}

// Prefill workspace: per-row metadata (4 int32 arrays of n) then the decode
// workspace of the n virtual one-query requests.
struct PrefillWs {
    int32_t *pos, *sid, *vlen, *req_row;
    void *dec;
    size_t dec_bytes, bytes;
};

static PrefillWs prefill_ws_layout(void *base, int n, int H, int d_h, int r, int max_ctx) {
    PrefillWs w;
    char *p = static_cast<char *>(base);
    size_t o = 0;
    const size_t arr = align256(sizeof(int32_t) * (size_t)std::max(n, 1));
    w.pos = reinterpret_cast<int32_t *>(p + o); o += arr;
    w.sid = reinterpret_cast<int32_t *>(p + o); o += arr;
    w.vlen = reinterpret_cast<int32_t *>(p + o); o += arr;
    w.req_row = reinterpret_cast<int32_t *>(p + o); o += arr;
    w.dec = p + o;
    w.dec_bytes = decode_ws_bytes(std::max(n, 1), H, d_h, r, std::max(max_ctx, 1));
    o += w.dec_bytes;
    w.bytes = o;
    return w;
}

}  // namespace lrkv

using namespace lrkv;

extern "C" {

int lrkv_version(void) { return 100; }

int lrkv_profile_enable(int on) {
    for (int k = 0; k < 3 && on; ++k) {
        Profiler &p = g_prof[k];
        if (p.created) continue;
        for (int i = 0; i < 2 * Profiler::kCap; ++i) {
            cudaError_t e = cudaEventCreate(&p.ev[i]);
            if (e != cudaSuccess) {
                for (int j = 0; j < i; ++j) cudaEventDestroy(p.ev[j]);
                return cuda_fail(e);
            }
        }
        p.created = true;
    }
    g_prof_on = on != 0;
    g_prof[0].n = g_prof[1].n = g_prof[2].n = 0;
    return LRKV_OK;
}

int lrkv_profile_read(int32_t which, double *total_ms, int32_t *launches) {
    if (!total_ms || !launches || which < 0 || which > 2) return LRKV_E_INVALID_ARG;
    Profiler &p = g_prof[which];
    *total_ms = 0.0;
    *launches = p.n;
    if (p.n > 0) {
        cudaError_t e = cudaEventSynchronize(p.ev[2 * p.n - 1]);
        if (e != cudaSuccess) return cuda_fail(e);
        for (int i = 0; i < p.n; ++i) {
            float ms = 0.f;
            e = cudaEventElapsedTime(&ms, p.ev[2 * i], p.ev[2 * i + 1]);
            if (e != cudaSuccess) return cuda_fail(e);
            *total_ms += ms;
        }
    }
    p.n = 0;
    return LRKV_OK;
}

int lrkv_last_cuda_error(void) { return g_last_cuda_error; }

const char *lrkv_status_string(int status) {
    switch (status) {
        case LRKV_OK: return "ok";
        case LRKV_E_INVALID_ARG: return "invalid argument";
        case LRKV_E_SHAPE: return "unsupported or inconsistent shape";
        case LRKV_E_DTYPE: return "unsupported dtype";
        case LRKV_E_BOUNDS: return "bound violated";
        case LRKV_E_WORKSPACE: return "workspace missing, misaligned or too small";
        case LRKV_E_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

int lrkv_prefill_kernel_kind(const lrkv_cache_t *cache) {
    if (!cache) return LRKV_E_INVALID_ARG;
    const int st = check_cache(cache);
    if (st) return st;
    return prefill_tc_covers(*cache) ? LRKV_PREFILL_TILED : LRKV_PREFILL_PER_ROW;
}

size_t lrkv_cache_bytes(int32_t H, int32_t d_h, int32_t r, int64_t tokens, int32_t dtype) {
    return lrkv_cache_bytes_grouped(H, d_h, r, 1, tokens, dtype);
}

size_t lrkv_cache_bytes_grouped(int32_t H, int32_t d_h, int32_t r, int32_t G, int64_t tokens,
                                int32_t dtype) {
    if (check_dims(H, d_h, r, dtype) || tokens < 0 || G < 1 || G > H || H % G) return 0;
    return (size_t)tokens * 2 * ((size_t)G * d_h + (size_t)H * r) * elem_bytes(dtype);
}

size_t lrkv_decode_workspace_bytes(int32_t B, int32_t H, int32_t d_h, int32_t r,
                                   int32_t max_seq_len, int32_t dtype) {
    if (check_dims(H, d_h, r, dtype) || B < 1 || max_seq_len < 1) return 0;
    return decode_ws_bytes(B, H, d_h, r, max_seq_len);
}

int lrkv_append(const void *X, const int32_t *positions, const int32_t *seq_ids, int32_t n,
                int32_t d, const void *W_S_K, const void *W_S_V, const void *U_K, const void *U_V,
                const lrkv_cache_t *cache, const int32_t *page_table, int32_t B, int32_t max_pages,
                int32_t *dev_status, lrkv_stream_t stream) {
    int st = check_append(X, positions, seq_ids, n, d, W_S_K, W_S_V, U_K, U_V, cache, page_table,
                          B, max_pages);
    if (st) return st;
    return run_append(X, positions, seq_ids, n, d, W_S_K, W_S_V, U_K, U_V, cache, page_table, B,
                      max_pages, dev_status, (cudaStream_t)stream);
}

int lrkv_decode(const void *q, const lrkv_cache_t *cache, const void *B_K, const void *B_V,
                const int32_t *seq_lens, const int32_t *page_table, int32_t B, int32_t max_pages,
                int32_t max_seq_len, void *out, void *workspace, size_t workspace_bytes,
                int32_t *dev_status, lrkv_stream_t stream) {
    int st = check_cache(cache);
    if (st) return st;
    if (B < 1 || max_pages < 1 || max_seq_len < 1) return LRKV_E_SHAPE;
    if ((int64_t)max_pages * cache->page_size > INT32_MAX / 2) return LRKV_E_SHAPE;
    if ((int64_t)max_seq_len > (int64_t)max_pages * cache->page_size) return LRKV_E_BOUNDS;
    if ((int64_t)B * max_seq_len > INT32_MAX / 2) return LRKV_E_SHAPE;
    if (!q || !B_K || !B_V || !seq_lens || !page_table || !out) return LRKV_E_INVALID_ARG;
    if (!aligned16(q) || !aligned16(B_K) || !aligned16(B_V) || !aligned16(out))
        return LRKV_E_INVALID_ARG;
    if (!workspace || !aligned256(workspace)) return LRKV_E_WORKSPACE;
    DecodeArgs a;
    a.q = q;
    a.cache = *cache;
    a.B_K = B_K;
    a.B_V = B_V;
    a.seq_lens = seq_lens;
    a.page_table = page_table;
    a.req_row = nullptr;
    a.B = B;
    a.max_pages = max_pages;
    a.max_seq_len = max_seq_len;
    a.out = out;
    a.status = dev_status;
    a.stream = (cudaStream_t)stream;
    return run_decode(a, workspace, workspace_bytes);
}

int lrkv_decode_noalloc(const void *q, const lrkv_cache_t *cache, const void *B_K,
                        const void *B_V, const int32_t *seq_lens, const int32_t *page_table,
                        int32_t B, int32_t max_pages, int32_t max_seq_len, void *out,
                        int32_t *dev_status, lrkv_stream_t stream) {
    // Same host checks as lrkv_decode, then the built-in scratch array stands
    // in for the caller's workspace.
    int st = check_cache(cache);
    if (st) return st;
    if (B < 1 || max_pages < 1 || max_seq_len < 1) return LRKV_E_SHAPE;
    if ((int64_t)max_pages * cache->page_size > INT32_MAX / 2) return LRKV_E_SHAPE;
    if ((int64_t)max_seq_len > (int64_t)max_pages * cache->page_size) return LRKV_E_BOUNDS;
    if ((int64_t)B * max_seq_len > INT32_MAX / 2) return LRKV_E_SHAPE;
    if (!q || !B_K || !B_V || !seq_lens || !page_table || !out) return LRKV_E_INVALID_ARG;
    if (!aligned16(q) || !aligned16(B_K) || !aligned16(B_V) || !aligned16(out))
        return LRKV_E_INVALID_ARG;
    if (decode_ws_bytes(B, cache->H, cache->d_h, cache->r, max_seq_len) >
        (size_t)LRKV_NOALLOC_SCRATCH_BYTES)
        return LRKV_E_WORKSPACE;
    cudaError_t e;
    void *scratch = noalloc_scratch_address(&e);
    if (!scratch) return cuda_fail(e);
    DecodeArgs a;
    a.q = q;
    a.cache = *cache;
    a.B_K = B_K;
    a.B_V = B_V;
    a.seq_lens = seq_lens;
    a.page_table = page_table;
    a.req_row = nullptr;
    a.B = B;
    a.max_pages = max_pages;
    a.max_seq_len = max_seq_len;
    a.out = out;
    a.status = dev_status;
    a.stream = (cudaStream_t)stream;
    return run_decode(a, scratch, (size_t)LRKV_NOALLOC_SCRATCH_BYTES);
}

// Decode-step workspace: the decode's (the append derives its rows' places
// from the lengths and needs none).
static size_t step_ws_bytes(int B, int H, int d_h, int r, int max_seq_len, size_t *dec_bytes) {
    const size_t dec = align256(decode_ws_bytes(B, H, d_h, r, max_seq_len));
    if (dec_bytes) *dec_bytes = dec;
    return dec;
}

size_t lrkv_decode_step_workspace_bytes(int32_t B, int32_t H, int32_t d_h, int32_t r,
                                        int32_t max_seq_len, int32_t dtype) {
    if (check_dims(H, d_h, r, dtype) || B < 1 || max_seq_len < 1) return 0;
    return step_ws_bytes(B, H, d_h, r, max_seq_len, nullptr);
}

// Host-side checks of a decode step (the append's, with positions and ids
// derived from the lengths, and the decode's).
static int check_step(const void *X, int32_t d, const void *W_S_K, const void *W_S_V,
                      const void *U_K, const void *U_V, const void *q, const lrkv_cache_t *cache,
                      const void *B_K, const void *B_V, const int32_t *seq_lens,
                      const int32_t *page_table, int32_t B, int32_t max_pages,
                      int32_t max_seq_len, const void *out) {
    int st = check_append(X, seq_lens, seq_lens, B, d, W_S_K, W_S_V, U_K, U_V, cache, page_table,
                          B, max_pages);
    if (st) return st;
    if (max_seq_len < 1) return LRKV_E_SHAPE;
    if ((int64_t)max_seq_len > (int64_t)max_pages * cache->page_size) return LRKV_E_BOUNDS;
    if ((int64_t)B * max_seq_len > INT32_MAX / 2) return LRKV_E_SHAPE;
    if (!q || !B_K || !B_V || !out) return LRKV_E_INVALID_ARG;
    if (!aligned16(q) || !aligned16(B_K) || !aligned16(B_V) || !aligned16(out))
        return LRKV_E_INVALID_ARG;
    return LRKV_OK;
}

int lrkv_decode_step(const void *X, int32_t d, const void *W_S_K, const void *W_S_V,
                     const void *U_K, const void *U_V, const void *q, const lrkv_cache_t *cache,
                     const void *B_K, const void *B_V, const int32_t *seq_lens,
                     const int32_t *page_table, int32_t B, int32_t max_pages,
                     int32_t max_seq_len, void *out, void *workspace, size_t workspace_bytes,
                     int32_t *dev_status, lrkv_stream_t stream) {
    int st = check_step(X, d, W_S_K, W_S_V, U_K, U_V, q, cache, B_K, B_V, seq_lens, page_table, B,
                        max_pages, max_seq_len, out);
    if (st) return st;
    if (!workspace || !aligned256(workspace)) return LRKV_E_WORKSPACE;
    size_t dec_bytes = 0;
    if (workspace_bytes < step_ws_bytes(B, cache->H, cache->d_h, cache->r, max_seq_len, &dec_bytes))
        return LRKV_E_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    DecodeArgs a;
    a.q = q;
    a.cache = *cache;
    a.B_K = B_K;
    a.B_V = B_V;
    a.seq_lens = seq_lens;
    a.page_table = page_table;
    a.req_row = nullptr;
    a.B = B;
    a.max_pages = max_pages;
    a.max_seq_len = max_seq_len;
    a.out = out;
    a.status = dev_status;
    a.stream = s;
    // the append (and the key norms) place request b's row at seq_lens[b] - 1
    // themselves; the decode's prologue then overlaps them, since its inputs
    // are none of theirs
    st = run_append(X, nullptr, nullptr, B, d, W_S_K, W_S_V, U_K, U_V, cache, page_table, B,
                    max_pages, dev_status, s, seq_lens);
    if (st) return st;
    if (cache->N_K) {
        cudaError_t e = launch_key_norms(nullptr, nullptr, B, B_K, *cache, page_table, B, max_pages,
                                         dev_status, s, seq_lens);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    a.early = true;
    return run_decode(a, workspace, dec_bytes);
}

// Host-buffer decode step: the step's workspace, then device copies of X,
// q, seq_lens and out (256-byte aligned each).
struct HostStepWs {
    size_t step, x, q, lens, out, bytes;
};

static HostStepWs host_step_layout(int B, int H, int d_h, int r, int d, int max_seq_len,
                                   int dtype) {
    HostStepWs w;
    const size_t eb = dtype == LRKV_F32 ? 4 : 2;  // activations: fp32, else bf16
    size_t o = step_ws_bytes(B, H, d_h, r, max_seq_len, nullptr);
    w.step = o;
    w.x = o; o += align256((size_t)B * d * eb);
    w.q = o; o += align256((size_t)B * H * d_h * eb);
    w.lens = o; o += align256(sizeof(int32_t) * (size_t)B);
    w.out = o; o += align256((size_t)B * H * d_h * eb);
    w.bytes = o;
    return w;
}

// Device address of page-locked (or registered) host memory, if it has one;
// a failed lookup leaves no pending error behind.
static bool host_mapped(const void *p, void **dev) {
    *dev = nullptr;
    if (cudaHostGetDevicePointer(dev, const_cast<void *>(p), 0) != cudaSuccess) {
        (void)cudaGetLastError();
        *dev = nullptr;
        return false;
    }
    return *dev != nullptr;
}

static int check_host_step(const void *X_host, int32_t d, const void *W_S_K, const void *W_S_V,
                           const void *U_K, const void *U_V, const void *q_host,
                           const lrkv_cache_t *cache, const void *B_K, const void *B_V,
                           const int32_t *seq_lens_host, const int32_t *page_table, int32_t B,
                           int32_t max_pages, int32_t max_seq_len, const void *out_host,
                           const void *workspace, size_t workspace_bytes) {
    if (!X_host || !q_host || !seq_lens_host || !out_host) return LRKV_E_INVALID_ARG;
    if (!workspace || !aligned256(workspace)) return LRKV_E_WORKSPACE;
    // the device copies (256-byte aligned, inside the workspace) stand in for
    // the host buffers, which need no alignment
    int st = check_step(workspace, d, W_S_K, W_S_V, U_K, U_V, workspace, cache, B_K, B_V,
                        seq_lens_host, page_table, B, max_pages, max_seq_len, workspace);
    if (st) return st;
    if (workspace_bytes <
        host_step_layout(B, cache->H, cache->d_h, cache->r, d, max_seq_len, cache->dtype).bytes)
        return LRKV_E_WORKSPACE;
    return LRKV_OK;
}

size_t lrkv_decode_step_host_workspace_bytes(int32_t B, int32_t H, int32_t d_h, int32_t r,
                                             int32_t d, int32_t max_seq_len, int32_t dtype) {
    if (check_dims(H, d_h, r, dtype) || B < 1 || max_seq_len < 1 || d < 1 || d > 65536) return 0;
    return host_step_layout(B, H, d_h, r, d, max_seq_len, dtype).bytes;
}

int lrkv_decode_step_host(const void *X_host, int32_t d, const void *W_S_K, const void *W_S_V,
                          const void *U_K, const void *U_V, const void *q_host,
                          const lrkv_cache_t *cache, const void *B_K, const void *B_V,
                          const int32_t *seq_lens_host, const int32_t *page_table, int32_t B,
                          int32_t max_pages, int32_t max_seq_len, void *out_host, void *workspace,
                          size_t workspace_bytes, int32_t *dev_status, lrkv_stream_t stream) {
    int st = check_host_step(X_host, d, W_S_K, W_S_V, U_K, U_V, q_host, cache, B_K, B_V,
                             seq_lens_host, page_table, B, max_pages, max_seq_len, out_host,
                             workspace, workspace_bytes);
    if (st) return st;
    const HostStepWs w = host_step_layout(B, cache->H, cache->d_h, cache->r, d, max_seq_len,
                                          cache->dtype);
    char *base = static_cast<char *>(workspace);
    const size_t eb = cache->dtype == LRKV_F32 ? 4 : 2;
    const size_t x_bytes = (size_t)B * d * eb, q_bytes = (size_t)B * cache->H * cache->d_h * eb;
    cudaStream_t s = (cudaStream_t)stream;
    // page-locked buffers are read and written by the kernels through their
    // device-mapped addresses (one copy kernel stages the inputs, the decode's
    // last kernel writes out); other host memory goes through the copy engines
    void *mX, *mq, *ml, *mo;
    const bool in_mapped = host_mapped(X_host, &mX) && host_mapped(q_host, &mq) &&
                           host_mapped(seq_lens_host, &ml);
    const bool out_mapped = host_mapped(out_host, &mo) && aligned16(mo);
    cudaError_t e = cudaSuccess;
    if (in_mapped) {
        StageCopy c;
        c.src[0] = mX; c.dst[0] = base + w.x; c.bytes[0] = x_bytes;
        c.src[1] = mq; c.dst[1] = base + w.q; c.bytes[1] = q_bytes;
        c.src[2] = ml; c.dst[2] = base + w.lens; c.bytes[2] = sizeof(int32_t) * (size_t)B;
        e = launch_stage_copy(c, s);
    } else {
        e = cudaMemcpyAsync(base + w.x, X_host, x_bytes, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(base + w.q, q_host, q_bytes, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(base + w.lens, seq_lens_host, sizeof(int32_t) * (size_t)B,
                                cudaMemcpyHostToDevice, s);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    st = lrkv_decode_step(base + w.x, d, W_S_K, W_S_V, U_K, U_V, base + w.q, cache, B_K, B_V,
                          reinterpret_cast<const int32_t *>(base + w.lens), page_table, B, max_pages,
                          max_seq_len, out_mapped ? mo : base + w.out, workspace, w.step,
                          dev_status, stream);
    if (st || out_mapped) return st;
    e = cudaMemcpyAsync(out_host, base + w.out, q_bytes, cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? LRKV_OK : cuda_fail(e);
}

}  // extern "C"

struct lrkv_step_graph_s {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

extern "C" {

int lrkv_step_graph_create(lrkv_step_graph_t *graph, const void *X_host, int32_t d,
                           const void *W_S_K, const void *W_S_V, const void *U_K, const void *U_V,
                           const void *q_host, const lrkv_cache_t *cache, const void *B_K,
                           const void *B_V, const int32_t *seq_lens_host, const int32_t *page_table,
                           int32_t B, int32_t max_pages, int32_t max_seq_len, void *out_host,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status) {
    if (!graph) return LRKV_E_INVALID_ARG;
    *graph = nullptr;
    const int chk = check_host_step(X_host, d, W_S_K, W_S_V, U_K, U_V, q_host, cache, B_K, B_V,
                                    seq_lens_host, page_table, B, max_pages, max_seq_len, out_host,
                                    workspace, workspace_bytes);
    if (chk) return chk;
    // record on a private stream (relaxed mode: the launchers' one-time
    // kernel attribute calls run during the recording); a failed check ends
    // the capture before any node exists
    cudaStream_t cs;
    cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e);
    auto *g = new lrkv_step_graph_s;
    e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed);
    int st = e == cudaSuccess ? LRKV_OK : cuda_fail(e);
    if (st == LRKV_OK) {
        st = lrkv_decode_step_host(X_host, d, W_S_K, W_S_V, U_K, U_V, q_host, cache, B_K, B_V,
                                   seq_lens_host, page_table, B, max_pages, max_seq_len, out_host,
                                   workspace, workspace_bytes, dev_status, cs);
        e = cudaStreamEndCapture(cs, &g->graph);
        if (st == LRKV_OK && e != cudaSuccess) st = cuda_fail(e);
    }
    if (st == LRKV_OK) {
        e = cudaGraphInstantiate(&g->exec, g->graph, 0);
        if (e != cudaSuccess) st = cuda_fail(e);
    }
    cudaStreamDestroy(cs);
    if (st != LRKV_OK) {
        lrkv_step_graph_destroy(g);
        return st;
    }
    *graph = g;
    return LRKV_OK;
}

int lrkv_step_graph_launch(lrkv_step_graph_t graph, lrkv_stream_t stream) {
    if (!graph || !graph->exec) return LRKV_E_INVALID_ARG;
    const cudaError_t e = cudaGraphLaunch(graph->exec, (cudaStream_t)stream);
    return e == cudaSuccess ? LRKV_OK : cuda_fail(e);
}

void lrkv_step_graph_destroy(lrkv_step_graph_t graph) {
    if (!graph) return;
    if (graph->exec) cudaGraphExecDestroy(graph->exec);
    if (graph->graph) cudaGraphDestroy(graph->graph);
    delete graph;
}

size_t lrkv_prefill_workspace_bytes(int32_t B, int32_t n, int32_t H, int32_t d_h, int32_t r,
                                    int32_t max_ctx, int32_t dtype) {
    if (check_dims(H, d_h, r, dtype) || B < 1 || n < 0 || max_ctx < 1) return 0;
    return prefill_ws_layout(nullptr, n, H, d_h, r, max_ctx).bytes;
}

static int prefill_impl(const void *X, const void *Q, const int32_t *cu_rows,
                        const int32_t *start_pos, int32_t B, int32_t n, int32_t max_ctx, int32_t d,
                        const void *W_S_K, const void *W_S_V, const void *U_K, const void *U_V,
                        const void *B_K, const void *B_V, const lrkv_cache_t *cache,
                        const int32_t *page_table, int32_t max_pages, const float *rope,
                        int32_t rope_max_pos, void *out, void *workspace, size_t workspace_bytes,
                        int32_t *dev_status, lrkv_stream_t stream) {
    int st = check_append(X, cu_rows, start_pos, n, d, W_S_K, W_S_V, U_K, U_V, cache, page_table,
                          B, max_pages);
    if (st) return st;
    if (max_ctx < 1) return LRKV_E_SHAPE;
    if ((int64_t)max_ctx > (int64_t)max_pages * cache->page_size) return LRKV_E_BOUNDS;
    if (n == 0) return LRKV_OK;
    if ((int64_t)n * max_ctx > INT32_MAX / 2) return LRKV_E_SHAPE;
    if (!Q || !B_K || !B_V || !out || !aligned16(Q) || !aligned16(B_K) || !aligned16(B_V) ||
        !aligned16(out))
        return LRKV_E_INVALID_ARG;
    if (!workspace || !aligned256(workspace)) return LRKV_E_WORKSPACE;
    PrefillWs w = prefill_ws_layout(workspace, n, cache->H, cache->d_h, cache->r, max_ctx);
    if (workspace_bytes < w.bytes) return LRKV_E_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_prefill_rows(cu_rows, start_pos, B, n, max_pages * cache->page_size,
                                        w.pos, w.sid, w.vlen, w.req_row, dev_status, s);
    if (e != cudaSuccess) return cuda_fail(e);
    st = run_append(X, w.pos, w.sid, n, d, W_S_K, W_S_V, U_K, U_V, cache, page_table, B, max_pages,
                    dev_status, s);
    if (st) return st;
    if (cache->N_K) {
        e = launch_key_norms(w.pos, w.sid, n, B_K, *cache, page_table, B, max_pages, dev_status, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (!rope && !cache->N_K) {
        // Causal attention on tensor cores (query tiles of 128 rows per head).
        PrefillTcArgs p;
        p.Q = Q;
        p.cu_rows = cu_rows;
        p.start_pos = start_pos;
        p.B = B;
        p.n = n;
        p.max_ctx = max_ctx;
        p.B_K = B_K;
        p.B_V = B_V;
        p.cache = *cache;
        p.page_table = page_table;
        p.max_pages = max_pages;
        p.out = out;
        p.status = dev_status;
        p.stream = s;
        prof_before(LRKV_PROFILE_ATTENTION, s);
        const int rc = launch_prefill_tc(p);
        if (rc == 0) prof_after(LRKV_PROFILE_ATTENTION, s);
        if (rc < 0) return cuda_fail((cudaError_t)(-rc));
        if (rc == 0) return LRKV_OK;
    }
    // Other shapes: row i is a one-query decode over its request's rows
    // 0..pos_i, reading the page-table row of its request.
    DecodeArgs a;
    a.q = Q;
    a.cache = *cache;
    a.B_K = B_K;
    a.B_V = B_V;
    a.seq_lens = w.vlen;
    a.page_table = page_table;
    a.req_row = w.req_row;
    a.B = n;
    a.max_pages = max_pages;
    a.max_seq_len = max_ctx;
    a.out = out;
    a.status = dev_status;
    a.stream = s;
    a.rope = rope;
    a.rope_max_pos = rope_max_pos;
    return run_decode(a, w.dec, w.dec_bytes);
}

int lrkv_prefill(const void *X, const void *Q, const int32_t *cu_rows, const int32_t *start_pos,
                 int32_t B, int32_t n, int32_t max_ctx, int32_t d, const void *W_S_K,
                 const void *W_S_V, const void *U_K, const void *U_V, const void *B_K,
                 const void *B_V, const lrkv_cache_t *cache, const int32_t *page_table,
                 int32_t max_pages, void *out, void *workspace, size_t workspace_bytes,
                 int32_t *dev_status, lrkv_stream_t stream) {
    return prefill_impl(X, Q, cu_rows, start_pos, B, n, max_ctx, d, W_S_K, W_S_V, U_K, U_V, B_K,
                        B_V, cache, page_table, max_pages, nullptr, 0, out, workspace,
                        workspace_bytes, dev_status, stream);
}

// ---------------------------------------------------------------------------
// Exact rotary position embedding
// ---------------------------------------------------------------------------
static int check_rope(const lrkv_cache_t *cache, const void *table, int32_t max_pos, int32_t need) {
    if (cache->d_h % 2 || cache->r > kRopeMaxRank) return LRKV_E_SHAPE;
    if (!table || !aligned16(table)) return LRKV_E_INVALID_ARG;
    if (max_pos < need) return LRKV_E_BOUNDS;
    return LRKV_OK;
}

static size_t rope_table_bytes(int d_h, int max_pos) {
    return rope_table_f16_offset(d_h, max_pos) + sizeof(__half) * (size_t)max_pos * d_h;
}

// Decode workspace of lrkv_decode_rope: the decode workspace, then the
// tensor-core rotary path's operands and scores.
static size_t rope_ws_bytes(int B, int H, int d_h, int r, int max_seq_len, size_t *dec_bytes) {
    const size_t dec = align256(decode_ws_bytes(B, H, d_h, r, max_seq_len));
    if (dec_bytes) *dec_bytes = dec;
    return dec + rope_fast_ws_layout(nullptr, B, H, d_h, r, max_seq_len).bytes;
}

int lrkv_key_norms(const int32_t *positions, const int32_t *seq_ids, int32_t n, const void *B_K,
                   const lrkv_cache_t *cache, const int32_t *page_table, int32_t B,
                   int32_t max_pages, int32_t *dev_status, lrkv_stream_t stream) {
    int st = check_cache(cache);
    if (st) return st;
    if (!cache->N_K) return LRKV_E_INVALID_ARG;
    if (n < 0 || B < 1 || max_pages < 1) return LRKV_E_SHAPE;
    if ((int64_t)max_pages * cache->page_size > INT32_MAX / 2) return LRKV_E_SHAPE;
    if (n == 0) return LRKV_OK;
    if (!positions || !seq_ids || !B_K || !page_table || !aligned16(B_K)) return LRKV_E_INVALID_ARG;
    cudaError_t e = launch_key_norms(positions, seq_ids, n, B_K, *cache, page_table, B, max_pages,
                                     dev_status, (cudaStream_t)stream);
    return e == cudaSuccess ? LRKV_OK : cuda_fail(e);
}

size_t lrkv_rope_table_bytes(int32_t d_h, int32_t max_pos) {
    if (d_h < 2 || d_h > 256 || d_h % 2 || max_pos < 1 || max_pos > (1 << 24)) return 0;
    return rope_table_bytes(d_h, max_pos);
}

size_t lrkv_decode_rope_workspace_bytes(int32_t B, int32_t H, int32_t d_h, int32_t r,
                                        int32_t max_seq_len, int32_t dtype) {
    if (check_dims(H, d_h, r, dtype) || B < 1 || max_seq_len < 1) return 0;
    return rope_ws_bytes(B, H, d_h, r, max_seq_len, nullptr);
}

int lrkv_rope_table(double base, int32_t d_h, int32_t max_pos, void *table, lrkv_stream_t stream) {
    if (!(base > 1.0) || !std::isfinite(base)) return LRKV_E_INVALID_ARG;
    if (d_h < 2 || d_h > 256 || d_h % 2 || max_pos < 1 || max_pos > (1 << 24)) return LRKV_E_SHAPE;
    if (!table || !aligned16(table)) return LRKV_E_INVALID_ARG;
    cudaError_t e = launch_rope_table(base, d_h, max_pos, table, (cudaStream_t)stream);
    return e == cudaSuccess ? LRKV_OK : cuda_fail(e);
}

int lrkv_decode_rope(const void *q, const lrkv_cache_t *cache, const void *B_K, const void *B_V,
                     const int32_t *seq_lens, const int32_t *page_table, int32_t B,
                     int32_t max_pages, int32_t max_seq_len, const void *rope_table,
                     int32_t rope_max_pos, void *out, void *workspace, size_t workspace_bytes,
                     int32_t *dev_status, lrkv_stream_t stream) {
    int st = check_cache(cache);
    if (st) return st;
    if (B < 1 || max_pages < 1 || max_seq_len < 1) return LRKV_E_SHAPE;
    if ((int64_t)max_pages * cache->page_size > INT32_MAX / 2) return LRKV_E_SHAPE;
    if ((int64_t)max_seq_len > (int64_t)max_pages * cache->page_size) return LRKV_E_BOUNDS;
    if ((int64_t)B * max_seq_len > INT32_MAX / 2) return LRKV_E_SHAPE;
    if (!q || !B_K || !B_V || !seq_lens || !page_table || !out) return LRKV_E_INVALID_ARG;
    if (!aligned16(q) || !aligned16(B_K) || !aligned16(B_V) || !aligned16(out))
        return LRKV_E_INVALID_ARG;
    if ((st = check_rope(cache, rope_table, rope_max_pos, max_seq_len))) return st;
    if (!workspace || !aligned256(workspace)) return LRKV_E_WORKSPACE;
    size_t dec_bytes = 0;
    if (workspace_bytes < rope_ws_bytes(B, cache->H, cache->d_h, cache->r, max_seq_len, &dec_bytes))
        return LRKV_E_WORKSPACE;
    DecodeArgs a;
    a.q = q;
    a.cache = *cache;
    a.B_K = B_K;
    a.B_V = B_V;
    a.seq_lens = seq_lens;
    a.page_table = page_table;
    a.req_row = nullptr;
    a.B = B;
    a.max_pages = max_pages;
    a.max_seq_len = max_seq_len;
    a.out = out;
    a.status = dev_status;
    a.stream = (cudaStream_t)stream;
    a.rope = static_cast<const float *>(rope_table);
    a.rope16 = reinterpret_cast<const __half *>(static_cast<const char *>(rope_table) +
                                                rope_table_f16_offset(cache->d_h, rope_max_pos));
    a.rope_max_pos = rope_max_pos;
    if (rope_fast_supported(cache->H, cache->d_h, cache->r, cache->page_size, cache->dtype) &&
        !cache->N_K && cache_groups(*cache) == 1)
        a.rope_ws = rope_fast_ws_layout(static_cast<char *>(workspace) + dec_bytes, B, cache->H,
                                        cache->d_h, cache->r, max_seq_len);
    return run_decode(a, workspace, dec_bytes);
}

int lrkv_prefill_rope(const void *X, const void *Q, const int32_t *cu_rows,
                      const int32_t *start_pos, int32_t B, int32_t n, int32_t max_ctx, int32_t d,
                      const void *W_S_K, const void *W_S_V, const void *U_K, const void *U_V,
                      const void *B_K, const void *B_V, const lrkv_cache_t *cache,
                      const int32_t *page_table, int32_t max_pages, const void *rope_table,
                      int32_t rope_max_pos, void *out, void *workspace, size_t workspace_bytes,
                      int32_t *dev_status, lrkv_stream_t stream) {
    int st = check_cache(cache);
    if (st) return st;
    if ((st = check_rope(cache, rope_table, rope_max_pos, max_ctx))) return st;
    return prefill_impl(X, Q, cu_rows, start_pos, B, n, max_ctx, d, W_S_K, W_S_V, U_K, U_V, B_K,
                        B_V, cache, page_table, max_pages, static_cast<const float *>(rope_table),
                        rope_max_pos, out, workspace, workspace_bytes, dev_status, stream);
}

}  // extern "C"
