// LRKV cache append, generic path (any supported shape, fp32 or bf16).
//
// Reading note "Low-Rank Key Value Attention", section 3, Algorithm 1: the
// new rows X are projected once through the packed weight
// [W_S_K | W_S_V | U_K(all heads) | U_V(all heads)] and each row's four blocks
// are written at its token position, into the page the page table gives for
// (request, position / page_size), slot position % page_size, under the same
// page id in all four pools.
#include "append_kernels.cuh"

#include <algorithm>

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

// The same for row i of an append: its (request, position) from the step's
// lengths or from the caller's arrays.
template <typename T>
__device__ __forceinline__ int64_t append_dest_row(const AppendArgsT<T> &a, int i) {
    if (a.step_lens) {
        const int32_t L = a.step_lens[i];
        const int32_t b = i, pos = (L < 1 || L > a.step_max_len) ? -1 : L - 1;
        return append_dest_row(&pos, &b, 0, a.page_table, a.B, a.max_pages, a.num_pages,
                               a.page_size, a.status);
    }
    return append_dest_row(a.positions, a.seq_ids, i, a.page_table, a.B, a.max_pages, a.num_pages,
                           a.page_size, a.status);
}

constexpr int kAM = 32, kAN = 64, kAK = 32;

template <typename T>
__global__ void __launch_bounds__(256) append_generic_kernel(AppendArgsT<T> a) {
    __shared__ float Xs[kAK][kAM + 1];
    __shared__ float Ws[kAK][kAN + 1];
    __shared__ int64_t dst_row[kAM];
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const int c0 = blockIdx.x * kAN, i0 = blockIdx.y * kAM;
    const int d_h = a.d_h, Hr = a.H * a.r;
    const int Ntot = 2 * d_h + 2 * Hr;

    if (tid < kAM) {
        const int i = i0 + tid;
        dst_row[tid] = (i < a.n) ? append_dest_row(a, i) : -1;
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
            store_projected(a, (size_t)row, c, acc[rr][q]);
        }
    }
}

template <typename T>
cudaError_t launch_append_generic(const AppendArgsT<T> &a) {
    const int Ntot = 2 * a.d_h + 2 * a.H * a.r;
    dim3 grid((Ntot + kAN - 1) / kAN, (a.n + kAM - 1) / kAM);
    return launch_pdl(append_generic_kernel<T>, grid, dim3(256), 0, a.stream, a);
}

template cudaError_t launch_append_generic<float>(const AppendArgsT<float> &);
template cudaError_t launch_append_generic<__nv_bfloat16>(const AppendArgsT<__nv_bfloat16> &);

// ---------------------------------------------------------------------------
// Few-row append (one new row per request in a decode step).  The work is a
// skinny X[n x d] . W^T product bound by reading W once: a block holds up to
// 16 rows of X in shared memory and each warp streams two weight rows with
// 16-byte coalesced loads, accumulating in fp32.
// ---------------------------------------------------------------------------
constexpr int kSkRows = 16, kSkWarps = 4, kSkCols = 4;  // rows per block, warps, columns per warp

template <typename T>
__device__ __forceinline__ const T *weight_row(const AppendArgsT<T> &a, int c) {
    const int d_h = a.d_h, Hr = a.H * a.r;
    if (c < d_h) return a.W_S_K + (size_t)c * a.d;
    if (c < 2 * d_h) return a.W_S_V + (size_t)(c - d_h) * a.d;
    if (c < 2 * d_h + Hr) return a.U_K + (size_t)(c - 2 * d_h) * a.d;
    return a.U_V + (size_t)(c - 2 * d_h - Hr) * a.d;
}

template <typename T>
__global__ void __launch_bounds__(kSkWarps * 32) append_rows_kernel(AppendArgsT<T> a) {
    constexpr int V = Vec16<T>::N;  // elements per 16-byte chunk
    extern __shared__ __align__(16) unsigned char sk_raw[];
    T *xs = reinterpret_cast<T *>(sk_raw);  // [kSkRows][d]
    __shared__ int64_t dst_row[kSkRows];
    __shared__ __align__(8) uint64_t xbar;
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i0 = blockIdx.y * kSkRows;
    const int nr = min(kSkRows, a.n - i0);
    const int d = a.d;
    const int Ntot = 2 * a.d_h + 2 * a.H * a.r;
    const int c0 = (blockIdx.x * kSkWarps + warp) * kSkCols;  // this warp's first output column
    const T *wrow[kSkCols];
#pragma unroll
    for (int cc = 0; cc < kSkCols; ++cc) wrow[cc] = weight_row(a, min(c0 + cc, Ntot - 1));
    const int nchunk = d / V;

    // the block's rows of X (contiguous) arrive by one bulk copy while the
    // first weight chunks are loaded
    if (tid == 0) {
        mbar_init(&xbar, 1);
        fence_barrier_init();
        const uint32_t bytes = (uint32_t)(nr * d * sizeof(T));
        mbar_arrive_expect_tx(&xbar, bytes);
        bulk_load(xs, a.X + (size_t)i0 * d, bytes, &xbar);
    }
    uint4 wn[kSkCols];
#pragma unroll
    for (int cc = 0; cc < kSkCols; ++cc)
        if (lane < nchunk) wn[cc] = *reinterpret_cast<const uint4 *>(wrow[cc] + (size_t)lane * V);
    if (tid < kSkRows)
        dst_row[tid] = (tid < nr) ? append_dest_row(a, i0 + tid) : -1;
    __syncthreads();
    if (!mbar_wait(&xbar, 0)) {
        status_or(a.status, LRKV_STATUS_TIMEOUT);
        return;
    }

    float acc[kSkCols][kSkRows];
#pragma unroll
    for (int cc = 0; cc < kSkCols; ++cc)
#pragma unroll
        for (int r = 0; r < kSkRows; ++r) acc[cc][r] = 0.f;
    for (int q = lane; q < nchunk; q += 32) {
        float w[kSkCols][V];
#pragma unroll
        for (int cc = 0; cc < kSkCols; ++cc) Vec16<T>::load(reinterpret_cast<const T *>(&wn[cc]), w[cc]);
        // prefetch the next chunks of the weight rows
        if (q + 32 < nchunk) {
#pragma unroll
            for (int cc = 0; cc < kSkCols; ++cc)
                wn[cc] = *reinterpret_cast<const uint4 *>(wrow[cc] + (size_t)(q + 32) * V);
        }
#pragma unroll
        for (int r = 0; r < kSkRows; ++r) {
            if (r < nr) {
                float x[V];
                Vec16<T>::load(xs + (size_t)r * d + (size_t)q * V, x);
#pragma unroll
                for (int cc = 0; cc < kSkCols; ++cc)
#pragma unroll
                    for (int e = 0; e < V; ++e) acc[cc][r] = fmaf(w[cc][e], x[e], acc[cc][r]);
            }
        }
    }
    const int d_h = a.d_h, Hr = a.H * a.r;
#pragma unroll
    for (int cc = 0; cc < kSkCols; ++cc) {
        float mine = 0.f;
#pragma unroll
        for (int r = 0; r < kSkRows; ++r) {
            float v = acc[cc][r];
#pragma unroll
            for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == r) mine = v;
        }
        const int c = c0 + cc;
        if (c >= Ntot || lane >= nr) continue;
        const int64_t row = dst_row[lane];
        if (row < 0) continue;
        store_projected(a, (size_t)row, c, mine);
    }
}

// ---------------------------------------------------------------------------
// Few-row append on tensor cores (bf16).  A block makes 16 output columns
// (two 8-column n-tiles) for 16 rows of X; its 16 warps split the
// contraction d into 32-wide chunks (chunk c goes to warp c mod 16).  In a
// chunk a lane needs four 16-byte runs, straight from global memory: X rows
// gq and gq + 8 and weight rows gq and 8 + gq, each at k = 8 tq .. 8 tq + 7.
// The chunk's two k-steps give both operands the same map from physical k
// to fragment slot (k-step s takes 8 tq + 4 s + {0, 1} for slots 2 tq, 2 tq + 1
// and 8 tq + 4 s + {2, 3} for slots 2 tq + 8, 2 tq + 9), so each dot product
// still pairs matching k and every operand load is one 16-byte access; a
// warp's whole share (four chunks at d = 2048) is in flight at once.
// Partial sums meet in shared memory in a fixed order and are scattered to
// the cache.
// ---------------------------------------------------------------------------
constexpr int kTcRows = 16, kTcCols = 16, kTcWarps = 16, kTcBatch = 4;

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int w) {
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

__global__ void __launch_bounds__(kTcWarps * 32, 1) append_rows_mma_kernel(AppendArgsT<__nv_bfloat16> a) {
    __shared__ float part[kTcWarps][kTcRows][kTcCols + 1];
    __shared__ int64_t dst_row[kTcRows];
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int i0 = blockIdx.y * kTcRows;
    const int nr = min(kTcRows, a.n - i0);
    const int Ntot = 2 * a.d_h + 2 * a.H * a.r;
    const int c0 = blockIdx.x * kTcCols;
    const int d = a.d, nch = d / 32;
    if (tid < kTcRows)
        dst_row[tid] = (tid < nr) ? append_dest_row(a, i0 + tid) : -1;
    const bool ok0 = gq < nr, ok1 = gq + 8 < nr;
    const __nv_bfloat16 *x0 = a.X + (size_t)(i0 + (ok0 ? gq : 0)) * d + 8 * tq;
    const __nv_bfloat16 *x1 = a.X + (size_t)(i0 + (ok1 ? gq + 8 : 0)) * d + 8 * tq;
    const __nv_bfloat16 *w0 = weight_row(a, min(c0 + gq, Ntot - 1)) + 8 * tq;
    const __nv_bfloat16 *w1 = weight_row(a, min(c0 + 8 + gq, Ntot - 1)) + 8 * tq;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int base = warp; base < nch; base += kTcBatch * kTcWarps) {
        uint4 xa[kTcBatch], xb[kTcBatch], wa[kTcBatch], wb[kTcBatch];
#pragma unroll
        for (int u = 0; u < kTcBatch; ++u) {
            const int ch = base + u * kTcWarps;
            xa[u] = xb[u] = wa[u] = wb[u] = zero;
            if (ch < nch) {
                const size_t k = (size_t)ch * 32;
                if (ok0) xa[u] = __ldg(reinterpret_cast<const uint4 *>(x0 + k));
                if (ok1) xb[u] = __ldg(reinterpret_cast<const uint4 *>(x1 + k));
                wa[u] = __ldg(reinterpret_cast<const uint4 *>(w0 + k));
                wb[u] = __ldg(reinterpret_cast<const uint4 *>(w1 + k));
            }
        }
#pragma unroll
        for (int u = 0; u < kTcBatch; ++u) {
            if (base + u * kTcWarps < nch) {
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const uint32_t av[4] = {word_of(xa[u], 2 * s), word_of(xb[u], 2 * s),
                                            word_of(xa[u], 2 * s + 1), word_of(xb[u], 2 * s + 1)};
                    mma_bf16_16816(c[0], av, word_of(wa[u], 2 * s), word_of(wa[u], 2 * s + 1));
                    mma_bf16_16816(c[1], av, word_of(wb[u], 2 * s), word_of(wb[u], 2 * s + 1));
                }
            }
        }
    }
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
        const int col = nb * 8 + 2 * tq;
        part[warp][gq][col] = c[nb][0];
        part[warp][gq][col + 1] = c[nb][1];
        part[warp][gq + 8][col] = c[nb][2];
        part[warp][gq + 8][col + 1] = c[nb][3];
    }
    __syncthreads();
    if (tid < kTcRows * kTcCols) {
        const int row = tid / kTcCols, cc = tid % kTcCols, cidx = c0 + cc;
        if (row < nr && cidx < Ntot) {
            const int64_t dr = dst_row[row];
            if (dr >= 0) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kTcWarps; ++w) v += part[w][row][cc];
                store_projected(a, (size_t)dr, cidx, v);
            }
        }
    }
}

bool rows_mma_append_fits(const AppendArgsT<__nv_bfloat16> &a) {
    return a.n <= 4 * kTcRows && a.d % 32 == 0;
}

cudaError_t launch_append_rows_mma(const AppendArgsT<__nv_bfloat16> &a) {
    const int Ntot = 2 * a.d_h + 2 * a.H * a.r;
    dim3 grid((Ntot + kTcCols - 1) / kTcCols, (a.n + kTcRows - 1) / kTcRows);
    return launch_pdl(append_rows_mma_kernel, grid, dim3(kTcWarps * 32), 0, a.stream, a);
}

template <typename T>
bool rows_append_fits(const AppendArgsT<T> &a) {
    return a.n <= 4 * kSkRows && (size_t)kSkRows * a.d * sizeof(T) <= 160 * 1024 &&
           a.d % Vec16<T>::N == 0;
}

template <typename T>
cudaError_t launch_append_rows(const AppendArgsT<T> &a) {
    const int Ntot = 2 * a.d_h + 2 * a.H * a.r;
    const int cols_per_block = kSkWarps * kSkCols;
    dim3 grid((Ntot + cols_per_block - 1) / cols_per_block, (a.n + kSkRows - 1) / kSkRows);
    const size_t sm = (size_t)kSkRows * a.d * sizeof(T);
    cudaError_t e = smem_limit_once(append_rows_kernel<T>, 160 * 1024);
    if (e != cudaSuccess) return e;
    return launch_pdl(append_rows_kernel<T>, grid, dim3(kSkWarps * 32), sm, a.stream, a);
}

template bool rows_append_fits<float>(const AppendArgsT<float> &);
template bool rows_append_fits<__nv_bfloat16>(const AppendArgsT<__nv_bfloat16> &);
template cudaError_t launch_append_rows<float>(const AppendArgsT<float> &);
template cudaError_t launch_append_rows<__nv_bfloat16>(const AppendArgsT<__nv_bfloat16> &);

// ---------------------------------------------------------------------------
// Prefill set-up: per new row, its request, position, visible length and the
// page-table row it reads (the request itself).
// ---------------------------------------------------------------------------
__global__ void prefill_rows_kernel(const int32_t *__restrict__ cu_rows,
                                    const int32_t *__restrict__ start_pos, int B, int n,
                                    int max_len, int32_t *pos, int32_t *sid, int32_t *vlen,
                                    int32_t *req_row, int32_t *status) {
    pdl_wait();
    pdl_launch_dependents();
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



// Decode step with host buffers: copies up to three page-locked host
// buffers (device-mapped addresses) into device memory in one launch, 16, 4
// or 2 bytes per access as the addresses and sizes allow.
__global__ void __launch_bounds__(256) stage_copy_kernel(StageCopy c) {
    pdl_wait();
    pdl_launch_dependents();
    const size_t t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t nth = (size_t)gridDim.x * blockDim.x;
#pragma unroll 1
    for (int k = 0; k < StageCopy::kMax; ++k) {
        const char *src = static_cast<const char *>(c.src[k]);
        char *dst = static_cast<char *>(c.dst[k]);
        const size_t n = c.bytes[k];
        const uintptr_t al = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | n;
        if (al % 16 == 0) {
            for (size_t i = t0; i < n / 16; i += nth)
                reinterpret_cast<uint4 *>(dst)[i] = reinterpret_cast<const uint4 *>(src)[i];
        } else if (al % 4 == 0) {
            for (size_t i = t0; i < n / 4; i += nth)
                reinterpret_cast<uint32_t *>(dst)[i] = reinterpret_cast<const uint32_t *>(src)[i];
        } else {
            for (size_t i = t0; i < n / 2; i += nth)
                reinterpret_cast<uint16_t *>(dst)[i] = reinterpret_cast<const uint16_t *>(src)[i];
        }
    }
}

cudaError_t launch_stage_copy(const StageCopy &c, cudaStream_t s) {
    size_t most = 0;
    for (int k = 0; k < StageCopy::kMax; ++k) most = c.bytes[k] > most ? c.bytes[k] : most;
    const unsigned blocks = (unsigned)std::min<size_t>(4 * (size_t)device_sm_count(),
                                                       std::max<size_t>(1, (most / 16 + 255) / 256));
    return launch_pdl(stage_copy_kernel, dim3(blocks), dim3(256), 0, s, c);
}

cudaError_t launch_prefill_rows(const int32_t *cu_rows, const int32_t *start_pos, int B, int n,
                                int max_len, int32_t *pos, int32_t *sid, int32_t *vlen,
                                int32_t *req_row, int32_t *status, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    return launch_pdl(prefill_rows_kernel, dim3((n + 255) / 256), dim3(256), 0, s, cu_rows,
                      start_pos, B, n, max_len, pos, sid, vlen, req_row, status);
}

// ---------------------------------------------------------------------------
// Joint key norms (reading note, section 8): for each appended row and head,
// 1 / sqrt(mean_d (s + z B_K[h]^T)_d^2 + eps) of the key the cache holds.
// One warp per (row, head): the private coordinates go to shared memory, lane
// d expands channels d, d + 32, ... against row d of B_K[h].
// ---------------------------------------------------------------------------
template <typename T, typename TC>
__global__ void __launch_bounds__(256) key_norms_kernel(
    const int32_t *__restrict__ positions, const int32_t *__restrict__ seq_ids, int n,
    const T *__restrict__ B_K, const TC *__restrict__ S_K, const TC *__restrict__ R_K,
    T *__restrict__ N_K, const int32_t *__restrict__ page_table, int B, int max_pages, int num_pages,
    int page_size, int H, int d_h, int r, float sk_scale, float rk_scale, float eps, int32_t *status,
    int groups, const int32_t *__restrict__ step_lens) {
    // groups: shared key/value groups; head h reads group h / (H / groups).
    // step_lens (decode step): row i is request i's row at step_lens[i] - 1.
    pdl_wait();
    pdl_launch_dependents();
    __shared__ float zs[8][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + warp;  // (row, head) pair; warp-uniform
    if (gw >= (int64_t)n * H) return;
    const int i = (int)(gw / H), h = (int)(gw % H);
    int32_t b, pos;
    if (step_lens) {
        const int32_t L = step_lens[i];
        b = i;
        pos = (L < 1 || (int64_t)L > (int64_t)max_pages * page_size) ? -1 : L - 1;
    } else {
        b = seq_ids[i];
        pos = positions[i];
    }
    if (b < 0 || b >= B || pos < 0 || (int64_t)pos >= (int64_t)max_pages * page_size) {
        if (lane == 0 && h == 0) status_or(status, LRKV_STATUS_BAD_ROW);
        return;
    }
    const int32_t page = page_table[(size_t)b * max_pages + pos / page_size];
    if (page < 0 || page >= num_pages) {
        if (lane == 0 && h == 0) status_or(status, LRKV_STATUS_BAD_PAGE);
        return;
    }
    const size_t prow = (size_t)page * page_size + pos % page_size;
    for (int k = lane; k < r; k += 32) zs[warp][k] = CacheLoad<TC>::load(R_K + (prow * H + h) * r + k) * rk_scale;
    __syncwarp();
    const T *bk = B_K + (size_t)h * d_h * r;
    float ss = 0.f;
    // rows of B_K[h] as 16-byte vectors (r is a multiple of the vector width
    // for every supported dtype and B_K is 16-byte aligned), all in flight
    constexpr int V = Vec16<T>::N;
    for (int d = lane; d < d_h; d += 32) {
        float kd = CacheLoad<TC>::load(S_K + (prow * groups + h / (H / groups)) * d_h + d) * sk_scale;
        const T *row = bk + (size_t)d * r;
        for (int k = 0; k < r; k += V) {
            float bv[V];
            Vec16<T>::load(row + k, bv);
#pragma unroll
            for (int e = 0; e < V; ++e) kd = fmaf(bv[e], zs[warp][k + e], kd);
        }
        ss = fmaf(kd, kd, ss);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) Elem<T>::store(N_K + prow * H + h, 1.f / sqrtf(ss / (float)d_h + eps));
}

cudaError_t launch_key_norms(const int32_t *positions, const int32_t *seq_ids, int n, const void *B_K,
                             const lrkv_cache_t &c, const int32_t *page_table, int B, int max_pages,
                             int32_t *status, cudaStream_t s, const int32_t *step_lens) {
    if (n <= 0) return cudaSuccess;
    const int64_t warps = (int64_t)n * c.H;
    const unsigned blocks = (unsigned)((warps + 7) / 8);
    if (c.dtype == LRKV_F32)
        return launch_pdl(key_norms_kernel<float, float>, dim3(blocks), dim3(256), 0, s, positions,
                          seq_ids, n, static_cast<const float *>(B_K), static_cast<const float *>(c.S_K),
                          static_cast<const float *>(c.R_K), static_cast<float *>(c.N_K), page_table, B,
                          max_pages, c.num_pages, c.page_size, c.H, c.d_h, c.r, 1.f, 1.f, c.norm_eps,
                          status, cache_groups(c), step_lens);
    if (c.dtype == LRKV_FP8_E4M3)
        return launch_pdl(key_norms_kernel<__nv_bfloat16, uint8_t>, dim3(blocks), dim3(256), 0, s,
                          positions, seq_ids, n, static_cast<const __nv_bfloat16 *>(B_K),
                          static_cast<const uint8_t *>(c.S_K), static_cast<const uint8_t *>(c.R_K),
                          static_cast<__nv_bfloat16 *>(c.N_K), page_table, B, max_pages, c.num_pages,
                          c.page_size, c.H, c.d_h, c.r, c.scale[0], c.scale[2], c.norm_eps, status,
                          cache_groups(c), step_lens);
    return launch_pdl(key_norms_kernel<__nv_bfloat16, __nv_bfloat16>, dim3(blocks), dim3(256), 0, s,
                      positions, seq_ids, n, static_cast<const __nv_bfloat16 *>(B_K),
                      static_cast<const __nv_bfloat16 *>(c.S_K), static_cast<const __nv_bfloat16 *>(c.R_K),
                      static_cast<__nv_bfloat16 *>(c.N_K), page_table, B, max_pages, c.num_pages,
                      c.page_size, c.H, c.d_h, c.r, 1.f, 1.f, c.norm_eps, status, cache_groups(c),
                      step_lens);
}

}  // namespace lrkv
