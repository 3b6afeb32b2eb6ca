// Internal interface between the C-ABI layer and the decode kernels.
#pragma once

#include "lrkv_common.cuh"

namespace lrkv {

struct DecodeArgs {
    const void *q;
    lrkv_cache_t cache;
    const void *B_K;
    const void *B_V;
    const int32_t *seq_lens;
    const int32_t *page_table;
    const int32_t *req_row;  // page-table row of request b (NULL: row b)
    int B;
    int max_pages;
    int max_seq_len;
    void *out;
    int32_t *status;
    cudaStream_t stream;
    // Exact rotary position embedding when rope != nullptr: the cos/sin table
    // [rope_max_pos][d_h / 2] of lrkv_rope_table, and its f16 copy.  With
    // rope_ws.wt set (lrkv_decode_rope on a tensor-core shape) the rotary
    // score kernel and the split kernel's given-score mode run; otherwise the
    // generic split kernel.
    const float *rope = nullptr;
    const __half *rope16 = nullptr;
    int rope_max_pos = 0;
    RopeFastWs rope_ws = {};
    // The prologue's predecessor in the stream is the same call's append
    // (lrkv_decode_step), which writes none of q, B_K, seq_lens, out or the
    // workspace, and which let it launch only after passing its own wait: the
    // prologue then lets the split kernel launch at once, does all its work
    // and waits for the append at its end, so the private queries and the
    // split kernel's first copies overlap the append.  The split kernel holds
    // back the copies of tiles that hold a new row until its own wait (which
    // the prologue's completion, and so the append's, releases).
    bool early = false;
};

// Longest sequence length a decode attends: what the page table can hold;
// on the tensor-core rotary path also no longer than the table and than
// max_seq_len (which sizes its score array).  Longer requests get a zero
// output and LRKV_STATUS_BAD_SEQLEN.
inline int decode_max_len(const DecodeArgs &a) {
    int m = a.max_pages * a.cache.page_size;
    if (a.rope_ws.wt) {
        m = m < a.rope_max_pos ? m : a.rope_max_pos;
        m = m < a.max_seq_len ? m : a.max_seq_len;
    }
    return m;
}

// Largest private width the rotary split kernel keeps in registers.
constexpr int kRopeMaxRank = 64;
cudaError_t launch_rope_table(double base, int d_h, int max_pos, void *table, cudaStream_t s);

// Rows the split kernels stream for a request of length L: none for an
// invalid length, else L.
__host__ __device__ __forceinline__ int32_t streamed_len(int32_t L, int max_len) {
    return (L < 1 || L > max_len) ? 0 : L;
}

// beside_split: the tensor-core split kernel follows (smaller prologue blocks).
template <typename T>
cudaError_t launch_prologue(const DecodeArgs &a, const DecodeWs &ws, int G, int tile_align,
                            bool beside_split);
template <typename T>
cudaError_t launch_split_generic(const DecodeArgs &a, const DecodeWs &ws, int G);
template <typename T>
cudaError_t launch_combine(const DecodeArgs &a, const DecodeWs &ws, int G);

// Tensor-core split kernel (bf16, d_h = 128, page_size % 16 == 0, selected
// (H, r) pairs).  `fast_decode_supported` says whether a shape is covered;
// `fast_decode_grid` is its CTA count on this device.
bool fast_decode_supported(int H, int d_h, int r, int page_size, int dtype, int groups = 1);

int fast_decode_grid(int H, int r);
cudaError_t launch_split_fast(const DecodeArgs &a, const DecodeWs &ws, int G);

// Exact RoPE on the tensor cores (bf16 cache, a tensor-core decode shape with
// H % 8 == 0): launch_rope_scores writes every visible row's score into
// a.rope_ws.sc; launch_split_fast (with a.rope_ws set) then streams only S_V,
// R_V and those scores.
bool rope_fast_supported(int H, int d_h, int r, int page_size, int dtype);
cudaError_t launch_rope_scores(const DecodeArgs &a, const DecodeWs &ws);

int device_sm_count();

// Device address of the built-in scratch array used by lrkv_decode_noalloc on
// the current device (nullptr and *err set on failure).
void *noalloc_scratch_address(cudaError_t *err);

}  // namespace lrkv
