// LRKV decode: prologue (private query + balanced schedule), a generic split
// kernel for any supported shape and dtype, and the split combine.
//
// Reading note "Low-Rank Key Value Attention", section 3, Algorithm 2 with
// equations 6 and 7: the private query p = q B_K[h] is formed once per step;
// every visible row j is scored as (q.S_K[j] + p.R_K[h,j]) / sqrt(d_h); one
// online softmax (running max and exp-sum, both value accumulators rescaled
// together when the max moves) reduces S_V and R_V[h] with the same weights;
// the private reduction is expanded once by B_V[h]^T at the end.
#include "decode_kernels.cuh"

namespace lrkv {

// ---------------------------------------------------------------------------
// Prologue: blocks [0, B*H) form p[b,h,:] = q[b,h,:] B_K[h]; the last block
// validates sequence lengths and writes the balanced plan (row offsets and
// the per-CTA chunk).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) decode_prologue_kernel(
    const T *__restrict__ q, const T *__restrict__ B_K, const int32_t *__restrict__ seq_lens,
    int B, int H, int d_h, int r, int max_len, int G, int tile_align, DecodeWs ws,
    int32_t *status) {
    const int tid = threadIdx.x;
    if (blockIdx.x == (unsigned)(B * H)) {
        // --- plan: exclusive scan of validated lengths ---
        __shared__ int32_t part[256];
        const int per = (B + blockDim.x - 1) / blockDim.x;
        const int lo = tid * per, hi = min(B, lo + per);
        int32_t s = 0;
        for (int b = lo; b < hi; ++b) {
            int32_t L = seq_lens[b];
            if (L < 1 || L > max_len) L = 0;
            s += L;
        }
        part[tid] = s;
        __syncthreads();
        if (tid == 0) {
            int32_t run = 0;
            for (int i = 0; i < (int)blockDim.x; ++i) {
                int32_t v = part[i];
                part[i] = run;
                run += v;
            }
            ws.plan->total = run;
            int32_t chunk = (run + G - 1) / G;
            chunk = max(chunk, tile_align);
            chunk = (chunk + tile_align - 1) / tile_align * tile_align;
            ws.plan->chunk = chunk;
            ws.off[B] = run;
        }
        __syncthreads();
        int32_t run = part[tid];
        bool bad = false;
        for (int b = lo; b < hi; ++b) {
            int32_t L = seq_lens[b];
            if (L < 1 || L > max_len) {
                L = 0;
                bad = true;
            }
            ws.off[b] = run;
            run += L;
        }
        if (bad) status_or(status, LRKV_STATUS_BAD_SEQLEN);
        return;
    }
    // --- private query ---
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    extern __shared__ float qs[];
    const T *qp = q + ((size_t)b * H + h) * d_h;
    for (int d = tid; d < d_h; d += blockDim.x) qs[d] = Elem<T>::load(qp + d);
    __syncthreads();
    const T *bk = B_K + (size_t)h * d_h * r;
    for (int k = tid; k < r; k += blockDim.x) {
        float acc = 0.f;
        for (int d = 0; d < d_h; ++d) acc = fmaf(qs[d], Elem<T>::load(bk + (size_t)d * r + k), acc);
        ws.p[((size_t)b * H + h) * r + k] = acc;
    }
}

// First request whose row range ends after global row x (off is nondecreasing).
__device__ __forceinline__ int find_request(const int32_t *off, int B, int32_t x) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (off[mid + 1] > x) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

// ---------------------------------------------------------------------------
// Generic split kernel: grid (G, H), one head per CTA, 128 threads.  Plain
// fp32 FMA; used for fp32 caches and for shapes the tensor-core path does not
// cover.
// ---------------------------------------------------------------------------
constexpr int kGenTile = 128;

template <typename T>
__global__ void __launch_bounds__(kGenTile) decode_split_generic_kernel(
    const T *__restrict__ q, const T *__restrict__ S_K, const T *__restrict__ S_V,
    const T *__restrict__ R_K, const T *__restrict__ R_V, const int32_t *__restrict__ page_table,
    const int32_t *__restrict__ req_row, int max_pages, int num_pages, int page_size, int B, int H, int d_h, int r,
    float scale_log2, DecodeWs ws, int32_t *status) {
    extern __shared__ float sm[];
    float *qs = sm;                 // d_h
    float *ps = qs + d_h;           // r
    float *w = ps + r;              // kGenTile weights
    int32_t *row = reinterpret_cast<int32_t *>(w + kGenTile);  // kGenTile pool rows
    __shared__ float red[kGenTile / 32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = blockIdx.x, h = blockIdx.y;
    const int32_t total = ws.plan->total, chunk = ws.plan->chunk;
    int32_t start = g * chunk;
    const int32_t end = min(total, start + chunk);
    if (start >= end) return;
    int b = find_request(ws.off, B, start);

    while (start < end) {
        while (ws.off[b + 1] <= start) ++b;
        const int32_t base = ws.off[b];
        const int32_t seg_end = min(end, ws.off[b + 1]);
        const int t_a = start - base, t_b = seg_end - base;

        const int32_t *pt = page_table + (size_t)(req_row ? req_row[b] : b) * max_pages;
        for (int d = tid; d < d_h; d += kGenTile) qs[d] = Elem<T>::load(q + ((size_t)b * H + h) * d_h + d);
        for (int k = tid; k < r; k += kGenTile) ps[k] = ws.p[((size_t)b * H + h) * r + k];
        __syncthreads();

        float m = -INFINITY, l = 0.f;
        float accS[2] = {0.f, 0.f}, accR[2] = {0.f, 0.f};
        for (int t0 = t_a; t0 < t_b; t0 += kGenTile) {
            const int j = t0 + tid;
            bool valid = j < t_b;
            float s = -INFINITY;
            int32_t prow = -1;
            if (valid) {
                int32_t page = pt[j / page_size];
                if (page < 0 || page >= num_pages) {
                    status_or(status, LRKV_STATUS_BAD_PAGE);
                    valid = false;
                } else {
                    prow = page * page_size + j % page_size;
                    const T *sk = S_K + (size_t)prow * d_h;
                    const T *rk = R_K + ((size_t)prow * H + h) * r;
                    float acc = 0.f;
                    for (int d = 0; d < d_h; ++d) acc = fmaf(qs[d], Elem<T>::load(sk + d), acc);
                    for (int k = 0; k < r; ++k) acc = fmaf(ps[k], Elem<T>::load(rk + k), acc);
                    s = acc * scale_log2;
                }
            }
            // tile max
            float mx = s;
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) red[warp] = mx;
            __syncthreads();
            float m_tile = red[0];
            for (int i = 1; i < kGenTile / 32; ++i) m_tile = fmaxf(m_tile, red[i]);
            __syncthreads();
            const float m_new = fmaxf(m, m_tile);
            float alpha = 1.f, e = 0.f;
            if (m_new != -INFINITY) {
                alpha = exp2f(m - m_new);
                e = valid ? exp2f(s - m_new) : 0.f;
            }
            w[tid] = e;
            row[tid] = valid ? prow : -1;
            float sum = e;
            for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) red[warp] = sum;
            __syncthreads();
            float l_tile = 0.f;
            for (int i = 0; i < kGenTile / 32; ++i) l_tile += red[i];
            l = l * alpha + l_tile;
            m = m_new;
            const int n = min(kGenTile, t_b - t0);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                accS[i] *= alpha;
                accR[i] *= alpha;
                const int d = tid + i * kGenTile;
                if (d < d_h) {
                    float a = accS[i];
                    for (int jj = 0; jj < n; ++jj) {
                        if (row[jj] < 0) continue;
                        a = fmaf(w[jj], Elem<T>::load(S_V + (size_t)row[jj] * d_h + d), a);
                    }
                    accS[i] = a;
                }
                if (d < r) {
                    float a = accR[i];
                    for (int jj = 0; jj < n; ++jj) {
                        if (row[jj] < 0) continue;
                        a = fmaf(w[jj], Elem<T>::load(R_V + ((size_t)row[jj] * H + h) * r + d), a);
                    }
                    accR[i] = a;
                }
            }
            __syncthreads();
        }
        const size_t slot = (size_t)b + g;
        if (tid == 0) {
            ws.ml[(slot * H + h) * 2 + 0] = m;
            ws.ml[(slot * H + h) * 2 + 1] = l;
        }
        float *acc = ws.acc + (slot * H + h) * (size_t)(d_h + r);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int d = tid + i * kGenTile;
            if (d < d_h) acc[d] = accS[i];
            if (d < r) acc[d_h + d] = accR[i];
        }
        start = seg_end;
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Combine: grid (H, B).  Log-sum-exp merge of the request's segments, then
// out = accS / L + (accR / L) B_V[h]^T  (equation 7, expansion done once).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(128) decode_combine_kernel(const T *__restrict__ B_V,
                                                             int B, int H, int d_h, int r,
                                                             DecodeWs ws, T *__restrict__ out) {
    extern __shared__ float cr[];  // r (normalised private reduction)
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int32_t o0 = ws.off[b], o1 = ws.off[b + 1];
    T *dst = out + ((size_t)b * H + h) * d_h;
    if (o1 <= o0) {
        for (int d = tid; d < d_h; d += blockDim.x) Elem<T>::store(dst + d, 0.f);
        return;
    }
    const int32_t chunk = ws.plan->chunk;
    const int g_lo = o0 / chunk, g_hi = (o1 - 1) / chunk;
    float M = -INFINITY;
    for (int g = g_lo; g <= g_hi; ++g) M = fmaxf(M, ws.ml[(((size_t)b + g) * H + h) * 2]);
    float L = 0.f;
    for (int g = g_lo; g <= g_hi; ++g) {
        const float *ml = ws.ml + (((size_t)b + g) * H + h) * 2;
        if (ml[0] != -INFINITY) L += exp2f(ml[0] - M) * ml[1];
    }
    const float invL = (L > 0.f) ? 1.f / L : 0.f;
    const int W = d_h + r;
    for (int k = tid; k < r; k += blockDim.x) {
        float a = 0.f;
        for (int g = g_lo; g <= g_hi; ++g) {
            const size_t s = ((size_t)b + g) * H + h;
            const float m = ws.ml[s * 2];
            if (m != -INFINITY) a = fmaf(exp2f(m - M), ws.acc[s * W + d_h + k], a);
        }
        cr[k] = a * invL;
    }
    __syncthreads();
    const T *bv = B_V + (size_t)h * d_h * r;
    for (int d = tid; d < d_h; d += blockDim.x) {
        float a = 0.f;
        for (int g = g_lo; g <= g_hi; ++g) {
            const size_t s = ((size_t)b + g) * H + h;
            const float m = ws.ml[s * 2];
            if (m != -INFINITY) a = fmaf(exp2f(m - M), ws.acc[s * W + d], a);
        }
        float o = a * invL;
        const T *row = bv + (size_t)d * r;
        for (int k = 0; k < r; ++k) o = fmaf(cr[k], Elem<T>::load(row + k), o);
        Elem<T>::store(dst + d, o);
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
template <typename T>
cudaError_t launch_prologue(const DecodeArgs &a, const DecodeWs &ws, int G, int tile_align) {
    const int blocks = a.B * a.cache.H + 1;
    const size_t sm = sizeof(float) * a.cache.d_h;
    decode_prologue_kernel<T><<<blocks, 256, sm, a.stream>>>(
        static_cast<const T *>(a.q), static_cast<const T *>(a.B_K), a.seq_lens, a.B, a.cache.H,
        a.cache.d_h, a.cache.r, a.max_pages * a.cache.page_size, G, tile_align, ws, a.status);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_split_generic(const DecodeArgs &a, const DecodeWs &ws, int G) {
    const auto &c = a.cache;
    const size_t sm = sizeof(float) * (c.d_h + c.r + kGenTile) + sizeof(int32_t) * kGenTile;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)c.d_h);
    dim3 grid(G, c.H);
    decode_split_generic_kernel<T><<<grid, kGenTile, sm, a.stream>>>(
        static_cast<const T *>(a.q), static_cast<const T *>(c.S_K), static_cast<const T *>(c.S_V),
        static_cast<const T *>(c.R_K), static_cast<const T *>(c.R_V), a.page_table, a.req_row, a.max_pages,
        c.num_pages, c.page_size, a.B, c.H, c.d_h, c.r, scale_log2, ws, a.status);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_combine(const DecodeArgs &a, const DecodeWs &ws) {
    dim3 grid(a.cache.H, a.B);
    decode_combine_kernel<T><<<grid, 128, sizeof(float) * a.cache.r, a.stream>>>(
        static_cast<const T *>(a.B_V), a.B, a.cache.H, a.cache.d_h, a.cache.r, ws,
        static_cast<T *>(a.out));
    return cudaGetLastError();
}

template cudaError_t launch_prologue<float>(const DecodeArgs &, const DecodeWs &, int, int);
template cudaError_t launch_prologue<__nv_bfloat16>(const DecodeArgs &, const DecodeWs &, int, int);
template cudaError_t launch_split_generic<float>(const DecodeArgs &, const DecodeWs &, int);
template cudaError_t launch_split_generic<__nv_bfloat16>(const DecodeArgs &, const DecodeWs &, int);
template cudaError_t launch_combine<float>(const DecodeArgs &, const DecodeWs &);
template cudaError_t launch_combine<__nv_bfloat16>(const DecodeArgs &, const DecodeWs &);

}  // namespace lrkv
