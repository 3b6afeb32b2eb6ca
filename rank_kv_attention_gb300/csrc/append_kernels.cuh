// Internal interface between the C-ABI layer and the append kernels.
#pragma once

#include "lrkv_common.cuh"

namespace lrkv {

template <typename T>
struct AppendArgsT {
    const T *X;
    const int32_t *positions;
    const int32_t *seq_ids;
    // decode step: when set, row i is request i's row at position
    // step_lens[i] - 1 (positions and seq_ids unused; a length outside
    // [1, step_max_len] skips the row and flags it)
    const int32_t *step_lens = nullptr;
    int step_max_len = 0;
    int n, d;
    const T *W_S_K, *W_S_V, *U_K, *U_V;
    T *S_K, *S_V, *R_K, *R_V;
    const int32_t *page_table;
    int B, max_pages, num_pages, page_size, H, d_h, r;
    int32_t *status;
    cudaStream_t stream;
    // LRKV_FP8_E4M3: the pools are 8-bit codes (S_K .. R_V above unused)
    bool fp8 = false;
    uint8_t *q8[4] = {nullptr, nullptr, nullptr, nullptr};  // S_K, S_V, R_K, R_V codes
    float inv_scale[4] = {1.f, 1.f, 1.f, 1.f};
};

// Store value v of packed output column c (0 .. 2 d_h + 2 H r) for pool row
// `row`: the four pools in order S_K, S_V, R_K, R_V.
template <typename T>
__device__ __forceinline__ void store_projected(const AppendArgsT<T> &a, size_t row, int c, float v) {
    const int Hr = a.H * a.r;
    int k, col;
    size_t width;
    if (c < a.d_h) { k = 0; col = c; width = a.d_h; }
    else if (c < 2 * a.d_h) { k = 1; col = c - a.d_h; width = a.d_h; }
    else if (c < 2 * a.d_h + Hr) { k = 2; col = c - 2 * a.d_h; width = Hr; }
    else { k = 3; col = c - 2 * a.d_h - Hr; width = Hr; }
    if (a.fp8) {
        a.q8[k][row * width + col] = (uint8_t)(e4m3x2_from_f32(v * a.inv_scale[k], 0.f) & 0xffu);
    } else {
        T *base = k == 0 ? a.S_K : k == 1 ? a.S_V : k == 2 ? a.R_K : a.R_V;
        Elem<T>::store(base + row * width + col, v);
    }
}

template <typename T>
cudaError_t launch_append_generic(const AppendArgsT<T> &a);

// Reciprocal joint key norms of n cached rows into c.N_K (see lrkv_key_norms).
cudaError_t launch_key_norms(const int32_t *positions, const int32_t *seq_ids, int n, const void *B_K,
                             const lrkv_cache_t &c, const int32_t *page_table, int B, int max_pages,
                             int32_t *status, cudaStream_t s, const int32_t *step_lens = nullptr);

// Few-row append (decode step): whether the shape fits, and the launcher.
template <typename T>
bool rows_append_fits(const AppendArgsT<T> &a);
template <typename T>
cudaError_t launch_append_rows(const AppendArgsT<T> &a);

// Few-row append on tensor cores (bf16): whether the shape fits, launcher.
bool rows_mma_append_fits(const AppendArgsT<__nv_bfloat16> &a);
cudaError_t launch_append_rows_mma(const AppendArgsT<__nv_bfloat16> &a);

// Tensor-core append (bf16): covered shapes and launcher.
bool tc_append_supported(int n, int d, int d_h, int H, int r);
cudaError_t launch_append_tc(const AppendArgsT<__nv_bfloat16> &a);
int device_sm_count();  // SMs of the current device (lrkv_api.cu)

// Up to three buffer copies (even byte counts) done by one kernel; unused
// entries have bytes = 0.
struct StageCopy {
    static constexpr int kMax = 3;
    const void *src[kMax] = {nullptr, nullptr, nullptr};
    void *dst[kMax] = {nullptr, nullptr, nullptr};
    size_t bytes[kMax] = {0, 0, 0};
};
cudaError_t launch_stage_copy(const StageCopy &c, cudaStream_t s);
cudaError_t launch_prefill_rows(const int32_t *cu_rows, const int32_t *start_pos, int B, int n,
                                int max_len, int32_t *pos, int32_t *sid, int32_t *vlen,
                                int32_t *req_row, int32_t *status, cudaStream_t s);

// Causal prefill attention on tensor cores (bf16, d_h = 128, r % 8 == 0,
// r <= 64, page_size % 64 == 0).  Returns 0 when launched, 1 when the shape
// is not covered (nothing enqueued), or -cudaError_t on a launch failure.
struct PrefillTcArgs {
    const void *Q;
    const int32_t *cu_rows, *start_pos;
    int B, n, max_ctx;
    const void *B_K, *B_V;
    lrkv_cache_t cache;
    const int32_t *page_table;
    int max_pages;
    void *out;
    int32_t *status;
    cudaStream_t stream;
};
int launch_prefill_tc(const PrefillTcArgs &p);
// Whether lrkv_prefill runs the tensor-core attention kernel for this cache.
bool prefill_tc_covers(const lrkv_cache_t &cache);

}  // namespace lrkv
