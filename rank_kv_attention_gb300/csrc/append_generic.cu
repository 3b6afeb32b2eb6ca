// LRKV cache append, generic path (any supported shape, fp32 or bf16).
//
// Reading note "Low-Rank Key Value Attention", section 3, Algorithm 1: the
// new rows X are projected once through the packed weight
// [W_S_K | W_S_V | U_K(all heads) | U_V(all heads)] and each row's four blocks
// are written at its token position, into the page the page table gives for
// (request, position / page_size), slot position % page_size, under the same
// page id in all four pools.
#include "append_kernels.cuh"

namespace lrkv {

// Destination pool row (page * page_size + slot) of append row i, or -1.
__device__ __forceinline__ int64_t append_dest_row(const int32_t *positions, const int32_t *seq_ids,
                                                   int i, const int32_t *page_table, int B,
                                                   int max_pages, int num_pages, int page_size,
                                                   int32_t *status) {
    const int32_t b = seq_ids[i], pos = positions[i];
    if (b < 0 || b >= B || pos < 0 || pos >= max_pages * page_size) {
        status_or(status, LRKV_STATUS_BAD_ROW);
        return -1;
    }
    const int32_t page = page_table[(size_t)b * max_pages + pos / page_size];
    if (page < 0 || page >= num_pages) {
        status_or(status, LRKV_STATUS_BAD_PAGE);
        return -1;
    }
    return (int64_t)page * page_size + pos % page_size;
}

constexpr int kAM = 32, kAN = 64, kAK = 32;

template <typename T>
__global__ void __launch_bounds__(256) append_generic_kernel(AppendArgsT<T> a) {
    __shared__ float Xs[kAK][kAM + 1];
    __shared__ float Ws[kAK][kAN + 1];
    __shared__ int64_t dst_row[kAM];
    const int tid = threadIdx.x;
    const int c0 = blockIdx.x * kAN, i0 = blockIdx.y * kAM;
    const int d_h = a.d_h, Hr = a.H * a.r;
    const int Ntot = 2 * d_h + 2 * Hr;

    if (tid < kAM) {
        const int i = i0 + tid;
        dst_row[tid] = (i < a.n) ? append_dest_row(a.positions, a.seq_ids, i, a.page_table, a.B,
                                                   a.max_pages, a.num_pages, a.page_size, a.status)
                                 : -1;
    }
    const int ty = tid / 16, tx = tid % 16;
    float acc[2][4] = {};
    for (int k0 = 0; k0 < a.d; k0 += kAK) {
        for (int e = tid; e < kAM * kAK; e += 256) {
            const int ii = e / kAK, kk = e % kAK;
            const int i = i0 + ii, k = k0 + kk;
            Xs[kk][ii] = (i < a.n && k < a.d) ? Elem<T>::load(a.X + (size_t)i * a.d + k) : 0.f;
        }
        for (int e = tid; e < kAN * kAK; e += 256) {
            const int cc = e / kAK, kk = e % kAK;
            const int c = c0 + cc, k = k0 + kk;
            float w = 0.f;
            if (c < Ntot && k < a.d) {
                const T *row;
                if (c < d_h) row = a.W_S_K + (size_t)c * a.d;
                else if (c < 2 * d_h) row = a.W_S_V + (size_t)(c - d_h) * a.d;
                else if (c < 2 * d_h + Hr) row = a.U_K + (size_t)(c - 2 * d_h) * a.d;
                else row = a.U_V + (size_t)(c - 2 * d_h - Hr) * a.d;
                w = Elem<T>::load(row + k);
            }
            Ws[kk][cc] = w;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kAK; ++kk) {
            const float x0 = Xs[kk][ty * 2], x1 = Xs[kk][ty * 2 + 1];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float w = Ws[kk][tx * 4 + q];
                acc[0][q] = fmaf(x0, w, acc[0][q]);
                acc[1][q] = fmaf(x1, w, acc[1][q]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int64_t row = dst_row[ty * 2 + rr];
        if (row < 0) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int c = c0 + tx * 4 + q;
            if (c >= Ntot) continue;
            T *dst;
            if (c < d_h) dst = a.S_K + row * d_h + c;
            else if (c < 2 * d_h) dst = a.S_V + row * d_h + (c - d_h);
            else if (c < 2 * d_h + Hr) dst = a.R_K + row * Hr + (c - 2 * d_h);
            else dst = a.R_V + row * Hr + (c - 2 * d_h - Hr);
            Elem<T>::store(dst, acc[rr][q]);
        }
    }
}

template <typename T>
cudaError_t launch_append_generic(const AppendArgsT<T> &a) {
    const int Ntot = 2 * a.d_h + 2 * a.H * a.r;
    dim3 grid((Ntot + kAN - 1) / kAN, (a.n + kAM - 1) / kAM);
    append_generic_kernel<T><<<grid, 256, 0, a.stream>>>(a);
    return cudaGetLastError();
}

template cudaError_t launch_append_generic<float>(const AppendArgsT<float> &);
template cudaError_t launch_append_generic<__nv_bfloat16>(const AppendArgsT<__nv_bfloat16> &);

// ---------------------------------------------------------------------------
// Prefill set-up: per new row, its request, position, visible length and the
// page-table row it reads (the request itself).
// ---------------------------------------------------------------------------
__global__ void prefill_rows_kernel(const int32_t *__restrict__ cu_rows,
                                    const int32_t *__restrict__ start_pos, int B, int n,
                                    int max_len, int32_t *pos, int32_t *sid, int32_t *vlen,
                                    int32_t *req_row, int32_t *status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    // request b with cu_rows[b] <= i < cu_rows[b+1]
    int lo = 0, hi = B;  // search in [0, B)
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (cu_rows[mid + 1] > i) hi = mid;
        else lo = mid + 1;
    }
    const int b = lo;
    bool ok = b < B && cu_rows[b] <= i && i < cu_rows[b + 1];
    int32_t p = ok ? start_pos[b] + (i - cu_rows[b]) : -1;
    if (ok && (p < 0 || p >= max_len)) ok = false;
    if (!ok) status_or(status, LRKV_STATUS_BAD_ROW);
    pos[i] = ok ? p : -1;
    sid[i] = ok ? b : -1;
    vlen[i] = ok ? p + 1 : 0;
    req_row[i] = ok ? b : 0;
}

cudaError_t launch_prefill_rows(const int32_t *cu_rows, const int32_t *start_pos, int B, int n,
                                int max_len, int32_t *pos, int32_t *sid, int32_t *vlen,
                                int32_t *req_row, int32_t *status, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    prefill_rows_kernel<<<(n + 255) / 256, 256, 0, s>>>(cu_rows, start_pos, B, n, max_len, pos, sid,
                                                         vlen, req_row, status);
    return cudaGetLastError();
}

}  // namespace lrkv
