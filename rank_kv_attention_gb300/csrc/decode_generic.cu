// LRKV decode: prologue (private query + balanced schedule), a generic split
// kernel for any supported shape and dtype, and the split combine.
//
// Reading note "Low-Rank Key Value Attention", section 3, Algorithm 2 with
// equations 6 and 7: the private query p = q B_K[h] is formed once per step;
// every visible row j is scored as (q.S_K[j] + p.R_K[h,j]) / sqrt(d_h); one
// online softmax (running max and exp-sum, both value accumulators rescaled
// together when the max moves) reduces S_V and R_V[h] with the same weights;
// the private reduction is expanded once by B_V[h]^T at the end.
#include <algorithm>
#include <type_traits>

#include "decode_kernels.cuh"

namespace lrkv {

// ---------------------------------------------------------------------------
// Prologue: block (x = h < H, y) forms p[b, h, :] = q[b, h, :] B_K[h] for the
// requests b of row group y, with B_K[h] staged in shared memory; block
// (x = H, y = 0) validates sequence lengths and writes the balanced plan (row
// offsets and rows per CTA).
// ---------------------------------------------------------------------------
constexpr int kProRows = 8;  // most requests per prologue block
constexpr size_t kStageFloats = 40 * 1024;  // largest B_K / B_V head staged in shared memory
constexpr int kProThreads = 256;  // threads of a prologue block

// Operands of the tensor-core rotary decode for head h of requests b0 ..
// b0 + nb - 1 (reading note, section 8).  With i = seq_len - 1 the query's
// position and q~ = q D_i its rotation, D_{i-j} = D_i D_j^T gives
//     (q D_{i-j}) B_K[h] = sum_c cos(j theta_c) A[c] + sin(j theta_c) Bq[c],
//     A[c][k]  = q~_2c B[2c][k] + q~_2c+1 B[2c+1][k],
//     Bq[c][k] = q~_2c+1 B[2c][k] - q~_2c B[2c+1][k],
// so the private query of key j is its (cos, sin) table row, interleaved by
// channel pair, times W = [A; Bq] interleaved the same way (row 2c = A[c],
// row 2c+1 = Bq[c]), and the shared term is q~ . (S_K[j] D_j).  Written per
// (b, h): q~ as a bf16 value row and a bf16 remainder row of the head group's
// block, and W transposed ([r][d_h], f16) after the exact power-of-two
// scaling that puts its largest |value| in [2^14, 2^15), with the inverse
// scale.  bk: B_K[h] as fp32 [d_h][r]; qs: the query rows; scratch: d_h +
// d_h r floats.
__device__ void rope_fast_operands(const float *bk, const float *qs, int nb, int b0, int h, int H,
                                   int d_h, int r, const int32_t *seq_lens, int max_len,
                                   const float2 *tab, const RopeFastWs &rf, float *scratch) {
    const int tid = threadIdx.x, hc = d_h / 2;
    float *qt = scratch, *w = scratch + d_h;
    __shared__ float wmax[kProThreads / 32];
    for (int bb = 0; bb < nb; ++bb) {
        const int b = b0 + bb;
        const int32_t L = seq_lens[b];
        if (L < 1 || L > max_len) continue;  // zeroed and flagged by the plan block
        const float2 *row = tab + (size_t)(L - 1) * hc;
        for (int c = tid; c < hc; c += blockDim.x) {
            const float2 cs = row[c];
            const float x0 = qs[bb * d_h + 2 * c], x1 = qs[bb * d_h + 2 * c + 1];
            const float y0 = x0 * cs.x - x1 * cs.y, y1 = x0 * cs.y + x1 * cs.x;
            qt[2 * c] = y0;
            qt[2 * c + 1] = y1;
        }
        {
            // this head's rows of the group block: bf16 value, bf16 remainder;
            // the group's first head also zeroes rows 2g .. 15
            const int g = rope_tc_heads_per_cta(r), i = h % g;
            uint16_t *blk = rf.qb + ((size_t)b * (H / g) + h / g) * 16 * d_h;
            __syncthreads();
            for (int c = tid; c < d_h; c += blockDim.x) {
                const __nv_bfloat16 hi = __float2bfloat16_rn(qt[c]);
                const __nv_bfloat16 lo = __float2bfloat16_rn(qt[c] - __bfloat162float(hi));
                blk[(size_t)i * d_h + c] = __bfloat16_as_ushort(hi);
                blk[(size_t)(g + i) * d_h + c] = __bfloat16_as_ushort(lo);
            }
            if (i == 0)
                for (int o = tid; o < (16 - 2 * g) * d_h; o += blockDim.x) blk[2 * g * d_h + o] = 0;
        }
        __syncthreads();
        float mx = 0.f;
        for (int o = tid; o < hc * r; o += blockDim.x) {
            const int c = o / r, k = o % r;
            const float u0 = bk[2 * c * r + k], u1 = bk[(2 * c + 1) * r + k];
            const float a = qt[2 * c] * u0 + qt[2 * c + 1] * u1;
            const float bq = qt[2 * c + 1] * u0 - qt[2 * c] * u1;
            w[2 * c * r + k] = a;
            w[(2 * c + 1) * r + k] = bq;
            mx = fmaxf(mx, fmaxf(fabsf(a), fabsf(bq)));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if ((tid & 31) == 0) wmax[tid >> 5] = mx;
        __syncthreads();
        mx = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) mx = fmaxf(mx, wmax[i]);
        const int e = f16_range_shift(mx);
        const float sc = exp2i(e);
        if (tid == 0) rf.wsc[(size_t)b * H + h] = exp2i(-e);
        // W^T: row n holds W[0 .. d_h)[n], two channels per 32-bit word
        const int nf = d_h * r / 2, hw = d_h / 2;
        uint32_t *dst = reinterpret_cast<uint32_t *>(rf.wt) + ((size_t)b * H + h) * nf;
        for (int f = tid; f < nf; f += blockDim.x) {
            const int n = f / hw, k0 = 2 * (f % hw);
            dst[f] = pack_f16(w[k0 * r + n] * sc, w[(k0 + 1) * r + n] * sc);
        }
        __syncthreads();  // qt, w and wmax are reused by the next request
    }
}

// ROPE: the exact-RoPE tensor-core operands instead of p (one request per
// block row).  NTHR: threads per block; 128-thread blocks (one request each,
// at most 51 registers a thread) fit on an SM beside a tensor-core split CTA.
template <typename T, bool ROPE, int NTHR>
__global__ void __launch_bounds__(NTHR, NTHR == 128 ? 10 : 1) decode_prologue_kernel(
    const T *__restrict__ q, const T *__restrict__ B_K, const int32_t *__restrict__ seq_lens,
    T *__restrict__ out,
    int B, int H, int d_h, int r, int max_len, int G, int tile_align, bool staged,
    DecodeWs ws, int32_t *status, const float2 *__restrict__ rope_tab, RopeFastWs rf, bool early) {
    constexpr int nrows = (ROPE || NTHR == 128) ? 1 : kProRows;
    const int tid = threadIdx.x;
    // early mode: the split kernel may launch at once (its own early work
    // reads none of this kernel's or the append's results, and it waits for
    // this grid before using them), and this block waits for the append as
    // it exits
    if (early) pdl_launch_dependents();
    const PdlWaitOnExit tail{early};
    if (!early && blockIdx.x < (unsigned)H) {
        // warm L2 with this block's B_K[h] and query rows while the
        // predecessor finishes: a prefetch reads nothing into the block, and
        // the loads below, after the wait, see every earlier write
        const char *bk = reinterpret_cast<const char *>(B_K + (size_t)blockIdx.x * d_h * r);
        const size_t bk_bytes = (size_t)d_h * r * sizeof(T);
        for (size_t o = (size_t)tid * 128; o < bk_bytes; o += (size_t)blockDim.x * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(bk + o));
        const int b_first = blockIdx.y * nrows;
        if (tid < nrows && b_first + tid < B) {
            const char *qr = reinterpret_cast<const char *>(q + ((size_t)(b_first + tid) * H + blockIdx.x) * d_h);
            for (size_t o = 0; o < (size_t)d_h * sizeof(T); o += 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(qr + o));
        }
    }
    if (!early) {
        pdl_wait();
        pdl_launch_dependents();
    }
    if (blockIdx.x == (unsigned)H) {
        // requests with an invalid length get a zero output (no segment will
        // ever write it)
        __shared__ int bad_len[kProRows];
        if (tid < nrows) {
            const int b = blockIdx.y * nrows + tid;
            int bad = 0;
            if (b < B) {
                const int32_t L = seq_lens[b];
                bad = (L < 1 || L > max_len);
            }
            bad_len[tid] = bad;
        }
        __syncthreads();
        for (int bb = 0; bb < nrows; ++bb)
            if (bad_len[bb])
                for (int i = tid; i < H * d_h; i += blockDim.x)
                    Elem<T>::store(out + (size_t)(blockIdx.y * nrows + bb) * H * d_h + i, 0.f);
        if (blockIdx.y != 0) return;
        // the tensor-core split kernel's counters
        if (tid < kDecodeCounters) ws.cnt[tid] = 0;
        // --- plan: exclusive scan of validated lengths ---
        __shared__ int32_t part[NTHR];
        const int per = (B + blockDim.x - 1) / blockDim.x;
        const int lo = tid * per, hi = min(B, lo + per);
        int32_t s = 0;
        for (int b = lo; b < hi; ++b) s += streamed_len(seq_lens[b], max_len);
        part[tid] = s;
        __syncthreads();
        constexpr int NPL = NTHR / 32;  // partial sums per lane
        if (tid < 32) {  // warp scan of the NTHR partial sums
            int32_t v[NPL], run = 0;
#pragma unroll
            for (int i = 0; i < NPL; ++i) { v[i] = part[tid * NPL + i]; run += v[i]; }
            int32_t incl = run;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += y;
            }
            int32_t ex = incl - run;
#pragma unroll
            for (int i = 0; i < NPL; ++i) { part[tid * NPL + i] = ex; ex += v[i]; }
            if (tid == 31) {
                ws.plan->total = incl;
                int32_t chunk = (incl + G - 1) / G;
                chunk = max(chunk, tile_align);
                chunk = (chunk + tile_align - 1) / tile_align * tile_align;
                ws.plan->chunk = chunk;
                ws.off[B] = incl;
            }
        }
        __syncthreads();
        int32_t run = part[tid];
        bool bad = false;
        for (int b = lo; b < hi; ++b) {
            const int32_t L = seq_lens[b];
            bad |= (L < 1 || L > max_len);
            ws.off[b] = run;
            run += streamed_len(L, max_len);
        }
        if (bad) status_or(status, LRKV_STATUS_BAD_SEQLEN);
        return;
    }
    // --- private queries of up to nrows requests for head h ---
    const int h = blockIdx.x, b0 = blockIdx.y * nrows;
    const int nb = min(nrows, B - b0);
    if constexpr (!ROPE && NTHR == 128 && sizeof(T) == 2) {
        if (d_h == 128 && (r & 7) == 0 && r <= 64) {
            // p = q B_K[h] of one request with every load in flight: warp w
            // sums channels 32 w .. 32 w + 31, lane o + 8 s (octet o < r/8 of
            // columns, slice s < 4 of eight channels) loads its eight 16-byte
            // B_K row slices and eight query values at once; xor-shuffles add
            // the slices and shared memory the warps, in a fixed order
            __shared__ float part[4][64];
            const int w = tid >> 5, lane = tid & 31, o = lane & 7, sl = lane >> 3;
            const int d0 = 32 * w + 8 * sl;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (8 * o < r) {
                const uint4 qv = *reinterpret_cast<const uint4 *>(q + ((size_t)b0 * H + h) * 128 + d0);
                uint4 bv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    bv[e] = *reinterpret_cast<const uint4 *>(B_K + ((size_t)h * 128 + d0 + e) * r + 8 * o);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t qw = (e >> 1) == 0 ? qv.x : (e >> 1) == 1 ? qv.y : (e >> 1) == 2 ? qv.z : qv.w;
                    const float qf = __uint_as_float((e & 1) ? (qw & 0xffff0000u) : (qw << 16));
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t bw = c == 0 ? bv[e].x : c == 1 ? bv[e].y : c == 2 ? bv[e].z : bv[e].w;
                        acc[2 * c] = fmaf(qf, __uint_as_float(bw << 16), acc[2 * c]);
                        acc[2 * c + 1] = fmaf(qf, __uint_as_float(bw & 0xffff0000u), acc[2 * c + 1]);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], 8);
                acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], 16);
            }
            if (sl == 0 && 8 * o < r)
#pragma unroll
                for (int c = 0; c < 8; ++c) part[w][8 * o + c] = acc[c];
            __syncthreads();
            if (tid < r)
                ws.p[((size_t)b0 * H + h) * r + tid] = (part[0][tid] + part[1][tid]) + (part[2][tid] + part[3][tid]);
            return;
        }
    }
    extern __shared__ float sm[];
    float *bk = sm;                               // [d_h][r] when staged
    float *qs = bk + (staged ? d_h * r : 0);      // [nrows][d_h]
    const T *src = B_K + (size_t)h * d_h * r;
    // query rows (one 16-byte vector per thread in flight) overlap the B_K staging
    constexpr int V = Vec16<T>::N;
    const int qv_row = d_h / V, nqv = nb * qv_row;
    float qv[V];
    const bool has_q = tid < nqv;
    if (has_q) Vec16<T>::load(q + ((size_t)(b0 + tid / qv_row) * H + h) * d_h + (tid % qv_row) * V, qv);
    if (staged) stage_f32(bk, src, d_h * r);
    if (has_q)
#pragma unroll
        for (int e = 0; e < V; ++e) qs[tid * V + e] = qv[e];
    for (int i = tid + blockDim.x; i < nqv; i += blockDim.x) {
        float v[V];
        Vec16<T>::load(q + ((size_t)(b0 + i / qv_row) * H + h) * d_h + (i % qv_row) * V, v);
#pragma unroll
        for (int e = 0; e < V; ++e) qs[i * V + e] = v[e];
    }
    __syncthreads();
    if constexpr (ROPE) {  // exact RoPE on the tensor cores: rotated queries and W
        rope_fast_operands(bk, qs, nb, b0, h, H, d_h, r, seq_lens, max_len, rope_tab, rf,
                           qs + nrows * d_h);
        return;
    }
    if (staged) {
        // four consecutive private columns per thread: per d one broadcast
        // query value, one 16-byte row slice of B_K[h] and four FMAs
        // (r % 4 == 0 for every supported dtype)
        const int r4 = r / 4;
        for (int o = tid; o < nb * r4; o += blockDim.x) {
            const int bb = o / r4, k = 4 * (o % r4);
            const float *qq = qs + bb * d_h;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
            int d = 0;
            for (; d + 1 < d_h; d += 2) {
                const float q0 = qq[d], q1 = qq[d + 1];
                const float4 b0 = *reinterpret_cast<const float4 *>(bk + d * r + k);
                const float4 b1 = *reinterpret_cast<const float4 *>(bk + (d + 1) * r + k);
                a.x = fmaf(q0, b0.x, a.x); a.y = fmaf(q0, b0.y, a.y);
                a.z = fmaf(q0, b0.z, a.z); a.w = fmaf(q0, b0.w, a.w);
                c.x = fmaf(q1, b1.x, c.x); c.y = fmaf(q1, b1.y, c.y);
                c.z = fmaf(q1, b1.z, c.z); c.w = fmaf(q1, b1.w, c.w);
            }
            if (d < d_h) {
                const float q0 = qq[d];
                const float4 b0 = *reinterpret_cast<const float4 *>(bk + d * r + k);
                a.x = fmaf(q0, b0.x, a.x); a.y = fmaf(q0, b0.y, a.y);
                a.z = fmaf(q0, b0.z, a.z); a.w = fmaf(q0, b0.w, a.w);
            }
            *reinterpret_cast<float4 *>(ws.p + ((size_t)(b0 + bb) * H + h) * r + k) =
                make_float4(a.x + c.x, a.y + c.y, a.z + c.z, a.w + c.w);
        }
    } else {
        for (int o = tid; o < nb * r; o += blockDim.x) {
            const int bb = o / r, k = o % r;
            const float *qq = qs + bb * d_h;
            float a0 = 0.f;
            for (int d = 0; d < d_h; ++d) a0 = fmaf(qq[d], Elem<T>::load(src + (size_t)d * r + k), a0);
            ws.p[((size_t)(b0 + bb) * H + h) * r + k] = a0;
        }
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

// Exact rotary position embedding (reading note, section 8).  The cache holds
// the unrotated projections; a key at position j meets a query at position i
// through D_i D_j^T = D_{i-j}, so with u = q D_{i-j} (channel pairs (2c, 2c+1)
// turned by (i - j) theta_c) its score is u.s_j + (u B_K[h]).z_j -- the
// note's (q~_i D_j^T B_h) z_j^T plus the rotated shared term.  Per (request,
// head) the kernel forms, for channel pair c and private column k,
//   A[c][k] = q_2c B[2c][k] + q_2c+1 B[2c+1][k],
//   Bq[c][k] = q_2c B[2c+1][k] - q_2c+1 B[2c][k],
// so that (u B_K[h])_k = sum_c cos(D theta_c) A[c][k] + sin(D theta_c) Bq[c][k]
// and u.s = sum_c cos (q_2c s_2c + q_2c+1 s_2c+1) + sin (q_2c s_2c+1 - q_2c+1 s_2c).
// cos and sin of D theta_c come from a table indexed by the distance D.
struct RopeArgs {
    const float2 *table;  // [max_pos][d_h / 2] (cos, sin)
    int max_pos;
};

// Private rotary scores of one 128-key tile on the tensor cores.  Warp w takes
// keys 32w .. 32w+31 of the tile as two 16-row m-tiles of
//     P[key][k] = sum over the interleaved (cos, sin) channels of the key's
//                 distance row times W[channel][k]   (f16 mma.sync, fp32 sum)
// then dots each row of P with that key's private coordinates and adds the
// result (scaled back by winv) to sh[key].  Keys whose row[] is -1 are not
// read (their MMA rows use distance 0 and are discarded).
template <typename TC, int RP>
__device__ __forceinline__ void rope_private_scores(const RopeArgs &rope, const __half *wt, int wstride,
                                                    const int32_t *row, float *sh, const TC *R_K, int H,
                                                    int h, int r, int d_h, int32_t q_pos, int t0,
                                                    float winv, int warp, int lane) {
    constexpr int NT = RP / 8;
    const int gq = lane >> 2, tq = lane & 3, hc = d_h / 2;
    float pacc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) pacc[mt][nt][e] = 0.f;
    const int mtx = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        const int r0 = 32 * warp + 16 * mt + gq, r1 = r0 + 8;
        const float2 *cs0 = rope.table + (size_t)(row[r0] >= 0 ? q_pos - (t0 + r0) : 0) * hc;
        const float2 *cs1 = rope.table + (size_t)(row[r1] >= 0 ? q_pos - (t0 + r1) : 0) * hc;
        for (int ks = 0; ks < d_h / 16; ++ks) {
            const int c0 = 8 * ks + tq, c1 = c0 + 4;
            const float2 e00 = cs0[c0], e10 = cs1[c0], e01 = cs0[c1], e11 = cs1[c1];
            const uint32_t a[4] = {pack_f16(e00.x, e00.y), pack_f16(e10.x, e10.y),
                                   pack_f16(e01.x, e01.y), pack_f16(e11.x, e11.y)};
#pragma unroll
            for (int nt = 0; nt < NT; nt += 2) {
                uint32_t b0, b1, b2, b3;
                const __half *src = wt + (8 * (nt + (mtx >> 1)) + rr) * wstride + 16 * ks + 8 * (mtx & 1);
                ldmatrix_x4(smem_u32(src), b0, b1, b2, b3);
                mma_f16_16816(pacc[mt][nt], a, b0, b1);
                mma_f16_16816(pacc[mt][nt + 1], a, b2, b3);
            }
        }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        const int r0 = 32 * warp + 16 * mt + gq, r1 = r0 + 8;
        const int32_t p0 = row[r0], p1 = row[r1];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = 8 * nt + 2 * tq;  // r is even: col < r implies col + 1 < r
            if (col < r) {
                if (p0 >= 0) {
                    const TC *z = R_K + ((size_t)p0 * H + h) * r + col;
                    s0 = fmaf(pacc[mt][nt][0], CacheLoad<TC>::load(z), s0);
                    s0 = fmaf(pacc[mt][nt][1], CacheLoad<TC>::load(z + 1), s0);
                }
                if (p1 >= 0) {
                    const TC *z = R_K + ((size_t)p1 * H + h) * r + col;
                    s1 = fmaf(pacc[mt][nt][2], CacheLoad<TC>::load(z), s1);
                    s1 = fmaf(pacc[mt][nt][3], CacheLoad<TC>::load(z + 1), s1);
                }
            }
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, o);
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        if (tq == 0) {
            if (p0 >= 0) sh[r0] += s0 * winv;
            if (p1 >= 0) sh[r1] += s1 * winv;
        }
    }
}

// T: query element type; TC: cache element type (T, or 8-bit codes whose pool
// scales sc = (S_K, S_V, R_K, R_V) fold into the queries and accumulators).
// RP > 0: scores with the exact rotary embedding, private width padded to RP.
template <typename T, typename TC, int RP = 0>
__global__ void __launch_bounds__(kGenTile) decode_split_generic_kernel(
    const T *__restrict__ q, const TC *__restrict__ S_K, const TC *__restrict__ S_V,
    const TC *__restrict__ R_K, const TC *__restrict__ R_V, const int32_t *__restrict__ page_table,
    const int32_t *__restrict__ req_row, int max_pages, int num_pages, int page_size, int B, int H, int d_h, int r,
    float scale_log2, float4 sc, DecodeWs ws, int32_t *status, const T *__restrict__ B_K, RopeArgs rope,
    const T *__restrict__ N_K, int s_stride, int hpg) {
    // s_stride: elements of a token's shared row (G d_h); hpg: heads per shared group
    extern __shared__ float sm[];
    float *qs = sm;                 // d_h
    float *ps = qs + d_h;           // r (plain) or A, Bq [d_h / 2][RP] each (rotary)
    float *w = ps + (RP ? d_h * RP : r);  // kGenTile weights
    int32_t *row = reinterpret_cast<int32_t *>(w + kGenTile);  // kGenTile pool rows
    // rotary on tensor cores (d_h % 16 == 0): per-key scores and the f16
    // coefficient matrix W^T [RP][d_h + 8] (rows padded for ldmatrix)
    float *sh = reinterpret_cast<float *>(row + kGenTile);
    __half *wt = reinterpret_cast<__half *>(sh + kGenTile);
    const int wstride = d_h + 8;
    // (bf16 activations only: f16 operands carry ~11 bits, the precision of
    // a bf16 result but not of the fp32 path)
    const bool use_mma = RP > 0 && d_h % 16 == 0 && !std::is_same<T, float>::value;
    float winv = 1.f;               // 2^-e of W's f16 scaling
    __shared__ float red[kGenTile / 32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = blockIdx.x, h = blockIdx.y;
    S_K += (size_t)(h / hpg) * d_h;  // this head's group of the shared rows
    S_V += (size_t)(h / hpg) * d_h;
    pdl_wait();
    pdl_launch_dependents();
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
        const int32_t q_pos = ws.off[b + 1] - base - 1;  // rotary: the query's position
        // rotary: a query past the end of the cos/sin table is not attended
        // (zero output, flagged) rather than read out of bounds
        const bool rope_ok = RP == 0 || q_pos < rope.max_pos;
        if (!rope_ok && tid == 0 && g * chunk <= base) status_or(status, LRKV_STATUS_BAD_SEQLEN);

        const int32_t *pt = page_table + (size_t)(req_row ? req_row[b] : b) * max_pages;
        const T *qr = q + ((size_t)b * H + h) * d_h;
        for (int d = tid; d < d_h; d += kGenTile) qs[d] = Elem<T>::load(qr + d) * sc.x;
        if constexpr (RP == 0) {
            for (int k = tid; k < r; k += kGenTile) ps[k] = ws.p[((size_t)b * H + h) * r + k] * sc.z;
        } else {
            // A and Bq of this (request, head), zero beyond column r; the R_K
            // pool scale folds in here
            const T *bk = B_K + (size_t)h * d_h * r;
            const int hc = d_h / 2;
            for (int i = tid; i < hc * RP; i += kGenTile) {
                const int c = i / RP, k = i % RP;
                float a = 0.f, bq = 0.f;
                if (k < r) {
                    const float q0 = Elem<T>::load(qr + 2 * c), q1 = Elem<T>::load(qr + 2 * c + 1);
                    const float b0 = Elem<T>::load(bk + (size_t)(2 * c) * r + k);
                    const float b1 = Elem<T>::load(bk + (size_t)(2 * c + 1) * r + k);
                    a = (q0 * b0 + q1 * b1) * sc.z;
                    bq = (q0 * b1 - q1 * b0) * sc.z;
                }
                ps[c * RP + k] = a;
                ps[hc * RP + c * RP + k] = bq;
            }
            if (use_mma) {
                // W[2c][k] = A[c][k], W[2c+1][k] = Bq[c][k], scaled by a power
                // of two into f16 range and stored transposed
                __syncthreads();
                float mx = 0.f;
                for (int i = tid; i < d_h * RP; i += kGenTile) mx = fmaxf(mx, fabsf(ps[i]));
#pragma unroll
                for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (lane == 0) red[warp] = mx;
                __syncthreads();
                mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
                const int e = f16_range_shift(mx);
                const float up = exp2i(e);
                winv = exp2i(-e);
                for (int i = tid; i < RP * d_h; i += kGenTile) {
                    const int k = i / d_h, dd = i % d_h, c = dd >> 1;
                    const float v = (dd & 1) ? ps[hc * RP + c * RP + k] : ps[c * RP + k];
                    wt[k * wstride + dd] = __float2half_rn(v * up);
                }
            }
        }
        __syncthreads();

        float m = -INFINITY, l = 0.f;
        float accS[2] = {0.f, 0.f}, accR[2] = {0.f, 0.f};
        for (int t0 = t_a; t0 < t_b; t0 += kGenTile) {
            const int j = t0 + tid;
            bool valid = j < t_b && rope_ok;
            float s = -INFINITY;
            int32_t prow = -1;
            if (valid) {
                int32_t page = pt[j / page_size];
                if (page < 0 || page >= num_pages) {
                    status_or(status, LRKV_STATUS_BAD_PAGE);
                    valid = false;
                } else {
                    prow = page * page_size + j % page_size;
                    const TC *sk = S_K + (size_t)prow * s_stride;
                    const TC *rk = R_K + ((size_t)prow * H + h) * r;
                    float acc = 0.f;
                    if constexpr (RP == 0) {
                        for (int d = 0; d < d_h; ++d) acc = fmaf(qs[d], CacheLoad<TC>::load(sk + d), acc);
                        for (int k = 0; k < r; ++k) acc = fmaf(ps[k], CacheLoad<TC>::load(rk + k), acc);
                    } else if (use_mma) {
                        // the rotated shared term here; the private term on
                        // the tensor cores below
                        const float2 *cs = rope.table + (size_t)(q_pos - j) * (d_h / 2);
                        for (int c = 0; c < d_h / 2; ++c) {
                            const float2 e = cs[c];
                            const float s0 = CacheLoad<TC>::load(sk + 2 * c);
                            const float s1 = CacheLoad<TC>::load(sk + 2 * c + 1);
                            const float q0 = qs[2 * c], q1 = qs[2 * c + 1];
                            acc = fmaf(e.x, fmaf(q0, s0, q1 * s1), acc);
                            acc = fmaf(e.y, fmaf(q0, s1, -q1 * s0), acc);
                        }
                    } else {
                        // distance from the query (the request's last row,
                        // which may lie beyond this segment) to key j
                        const float2 *cs = rope.table + (size_t)(q_pos - j) * (d_h / 2);
                        const int hc = d_h / 2;
                        float pk[RP];
#pragma unroll
                        for (int k = 0; k < RP; ++k) pk[k] = 0.f;
                        for (int c = 0; c < hc; ++c) {
                            const float2 e = cs[c];
                            const float s0 = CacheLoad<TC>::load(sk + 2 * c);
                            const float s1 = CacheLoad<TC>::load(sk + 2 * c + 1);
                            const float q0 = qs[2 * c], q1 = qs[2 * c + 1];
                            acc = fmaf(e.x, fmaf(q0, s0, q1 * s1), acc);
                            acc = fmaf(e.y, fmaf(q0, s1, -q1 * s0), acc);
                            const float *a = ps + c * RP, *bq = ps + hc * RP + c * RP;
#pragma unroll
                            for (int k = 0; k < RP; ++k) pk[k] = fmaf(e.x, a[k], fmaf(e.y, bq[k], pk[k]));
                        }
#pragma unroll
                        for (int k = 0; k < RP; ++k)
                            if (k < r) acc = fmaf(pk[k], CacheLoad<TC>::load(rk + k), acc);
                    }
                    if (use_mma) {
                        sh[tid] = acc;
                    } else {
                        if (N_K) acc *= Elem<T>::load(N_K + (size_t)prow * H + h);  // joint key norm
                        s = acc * scale_log2;
                    }
                }
            }
            if constexpr (RP > 0) {
                if (use_mma) {
                    row[tid] = valid ? prow : -1;
                    __syncthreads();
                    rope_private_scores<TC, RP>(rope, wt, wstride, row, sh, R_K, H, h, r, d_h, q_pos,
                                                t0, winv, warp, lane);
                    __syncthreads();
                    if (valid) {
                        float acc = sh[tid];
                        if (N_K) acc *= Elem<T>::load(N_K + (size_t)prow * H + h);  // joint key norm
                        s = acc * scale_log2;
                    }
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
                        a = fmaf(w[jj], CacheLoad<TC>::load(S_V + (size_t)row[jj] * s_stride + d), a);
                    }
                    accS[i] = a;
                }
                if (d < r) {
                    float a = accR[i];
                    for (int jj = 0; jj < n; ++jj) {
                        if (row[jj] < 0) continue;
                        a = fmaf(w[jj], CacheLoad<TC>::load(R_V + ((size_t)row[jj] * H + h) * r + d), a);
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
            if (d < d_h) acc[d] = accS[i] * sc.y;
            if (d < r) acc[d_h + d] = accR[i] * sc.w;
        }
        start = seg_end;
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Combine: grid (H, B), one block per (request, head).  Log-sum-exp merge of
// the request's segments, then out = accS / L + (accR / L) B_V[h]^T
// (equation 7, expansion done once).  All global reads (B_V[h], the
// segments' (m, l) and accumulators) are issued before the merge needs them.
// ---------------------------------------------------------------------------
constexpr int kCombSeg = 16;  // segments whose partials a thread keeps in flight

template <typename T>
__global__ void __launch_bounds__(256) decode_combine_kernel(const T *__restrict__ B_V,
                                                             int B, int H, int d_h, int r,
                                                             bool staged, DecodeWs ws,
                                                             T *__restrict__ out) {
    extern __shared__ __align__(16) float cs[];
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    // Until the wait below only a caller input is read (complete before the
    // prologue got past its own wait, which precedes this grid's launch):
    // B_V[h], staged in shared memory while the split kernel is still running.
    T *bv = reinterpret_cast<T *>(cs);                                   // [d_h][r] when staged
    const T *src = B_V + (size_t)h * d_h * r;
    const int nthr = blockDim.x, nwarp = nthr >> 5;
    if (staged) {
        const int nv = d_h * r * (int)sizeof(T) / 16;
        const uint4 *s16 = reinterpret_cast<const uint4 *>(src);
        uint4 *d16 = reinterpret_cast<uint4 *>(bv);
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (tid + u * nthr < nv) v[u] = s16[tid + u * nthr];
        for (int base = tid; base < nv; base += 4 * nthr) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (base + u * nthr < nv) d16[base + u * nthr] = v[u];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (base + (4 + u) * nthr < nv) v[u] = s16[base + (4 + u) * nthr];
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    const int32_t o0 = ws.off[b], o1 = ws.off[b + 1];
    T *dst = out + ((size_t)b * H + h) * d_h;
    if (o1 <= o0) {
        for (int d = tid; d < d_h; d += blockDim.x) Elem<T>::store(dst + d, 0.f);
        return;
    }
    const int32_t chunk = ws.plan->chunk;
    const int g_lo = o0 / chunk, nseg = (o1 - 1) / chunk - g_lo + 1;
    const int W = d_h + r;
    const size_t s0 = ((size_t)b + g_lo) * H + h;  // slot of segment g: s0 + g H
    float *cr = cs + (staged ? ((size_t)d_h * r * sizeof(T) + 15) / 16 * 4 : 0);  // [r]
    float *w = cr + r;                                                    // [nseg]
    __shared__ float red[2][8];
    // this thread's columns: c0 = tid, c1 = tid + blockDim.x (W <= 2 blockDim.x)
    const int c0 = tid, c1 = tid + nthr;
    float m_my = -INFINITY, l_my = 0.f;
    if (tid < nseg) {
        const float2 ml = *reinterpret_cast<const float2 *>(ws.ml + (s0 + (size_t)tid * H) * 2);
        m_my = ml.x;
        l_my = ml.y;
    }
    float a0 = 0.f, a1 = 0.f;
    float v0[kCombSeg], v1[kCombSeg];
#pragma unroll
    for (int g = 0; g < kCombSeg; ++g) {
        v0[g] = (g < nseg && c0 < W) ? ws.acc[(s0 + (size_t)g * H) * W + c0] : 0.f;
        v1[g] = (g < nseg && c1 < W) ? ws.acc[(s0 + (size_t)g * H) * W + c1] : 0.f;
    }
    // 2. merge weights
    float mx = m_my;
    for (int k = tid + nthr; k < nseg; k += nthr) mx = fmaxf(mx, ws.ml[(s0 + (size_t)k * H) * 2]);
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) red[0][tid >> 5] = mx;
    __syncthreads();
    float M = red[0][0];
    for (int i = 1; i < nwarp; ++i) M = fmaxf(M, red[0][i]);
    for (int k = tid; k < nseg; k += blockDim.x) {
        const float mk = (k == tid) ? m_my : ws.ml[(s0 + (size_t)k * H) * 2];
        w[k] = (mk == -INFINITY) ? 0.f : exp2f(mk - M);
    }
    float ls = (tid < nseg && m_my != -INFINITY) ? exp2f(m_my - M) * l_my : 0.f;
    for (int k = tid + nthr; k < nseg; k += blockDim.x) {
        const float2 ml = *reinterpret_cast<const float2 *>(ws.ml + (s0 + (size_t)k * H) * 2);
        if (ml.x != -INFINITY) ls = fmaf(exp2f(ml.x - M), ml.y, ls);
    }
    for (int o = 16; o; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    if ((tid & 31) == 0) red[1][tid >> 5] = ls;
    __syncthreads();
    float L = 0.f;
    for (int i = 0; i < nwarp; ++i) L += red[1][i];
    const float invL = (L > 0.f) ? 1.f / L : 0.f;
    // 3. weighted sums over segments
#pragma unroll
    for (int g = 0; g < kCombSeg; ++g) {
        if (g < nseg) {
            a0 = fmaf(w[g], v0[g], a0);
            a1 = fmaf(w[g], v1[g], a1);
        }
    }
    for (int g = kCombSeg; g < nseg; ++g) {
        const float *acc = ws.acc + (s0 + (size_t)g * H) * W;
        if (c0 < W) a0 = fmaf(w[g], acc[c0], a0);
        if (c1 < W) a1 = fmaf(w[g], acc[c1], a1);
    }
    a0 *= invL;
    a1 *= invL;
    // private part of the columns goes to shared memory for the expansion
    if (c0 >= d_h && c0 < W) cr[c0 - d_h] = a0;
    if (c1 >= d_h && c1 < W) cr[c1 - d_h] = a1;
    __syncthreads();
    // 4. out[d] = accS[d] / L + sum_k (accR[k] / L) B_V[h][d][k]
    for (int d = tid; d < d_h; d += blockDim.x) {
        float o = (d == c0) ? a0 : (d == c1) ? a1 : 0.f;
        if (staged) {
            const T *row = bv + (size_t)d * r;
            constexpr int V = Vec16<T>::N;
            for (int k = 0; k < r; k += V) {
                float x[V];
                Vec16<T>::load(row + k, x);
#pragma unroll
                for (int e = 0; e < V; ++e) o = fmaf(cr[k + e], x[e], o);
            }
        } else {
            const T *row = src + (size_t)d * r;
            for (int k = 0; k < r; ++k) o = fmaf(cr[k], Elem<T>::load(row + k), o);
        }
        Elem<T>::store(dst + d, o);
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
template <typename T>
cudaError_t launch_prologue(const DecodeArgs &a, const DecodeWs &ws, int G, int tile_align,
                            bool beside_split) {
    const auto &c = a.cache;
    // the rotary operands (W is d_h x r per request and head) take one 256-
    // thread block per (head, request); before the tensor-core split kernel,
    // p = q B_K runs in 128-thread blocks of one request each, which fit on
    // an SM beside a split CTA (so no split CTA waits for a prologue block to
    // leave); otherwise a block amortises B_K's staging over 8 requests
    const bool rope_fast = a.rope_ws.wt != nullptr;
    const bool small = !rope_fast && beside_split;
    const int nrows = (rope_fast || small) ? 1 : kProRows;
    dim3 grid(c.H + 1, (a.B + nrows - 1) / nrows);
    const bool staged = (size_t)c.d_h * c.r <= kStageFloats;
    const size_t sm = sizeof(float) * ((staged ? (size_t)c.d_h * c.r : 0) + (size_t)nrows * c.d_h +
                                       (rope_fast ? (size_t)c.d_h * (c.r + 1) : 0));
    // the tensor-core rotary path treats a request past the table's end as an
    // invalid length (zero output, flagged), like every kernel after it
    const int max_len = decode_max_len(a);
    auto kern = rope_fast ? decode_prologue_kernel<T, true, kProThreads>
              : small     ? decode_prologue_kernel<T, false, 128>
                          : decode_prologue_kernel<T, false, kProThreads>;
    cudaError_t e = smem_limit_once(kern, 200 * 1024);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, dim3(small ? 128 : kProThreads), sm, a.stream,
                      static_cast<const T *>(a.q), static_cast<const T *>(a.B_K), a.seq_lens,
                      static_cast<T *>(a.out), a.B, a.cache.H, a.cache.d_h, a.cache.r,
                      max_len, G, tile_align, staged, ws, a.status,
                      reinterpret_cast<const float2 *>(a.rope), a.rope_ws, a.early);
}

template <typename T, typename TC, int RP>
static cudaError_t launch_split_generic_t(const DecodeArgs &a, const DecodeWs &ws, int G) {
    const auto &c = a.cache;
    const size_t sm = sizeof(float) * (c.d_h + (RP ? (size_t)c.d_h * RP : c.r) + kGenTile) +
                      sizeof(int32_t) * kGenTile +
                      (RP ? sizeof(float) * kGenTile + sizeof(__half) * (size_t)RP * (c.d_h + 8) : 0);
    auto kern = decode_split_generic_kernel<T, TC, RP>;
    if (sm > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
    }
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)c.d_h);
    const bool q8 = c.dtype == LRKV_FP8_E4M3;
    const float4 sc = q8 ? make_float4(c.scale[0], c.scale[1], c.scale[2], c.scale[3])
                         : make_float4(1.f, 1.f, 1.f, 1.f);
    RopeArgs rope{reinterpret_cast<const float2 *>(a.rope), a.rope_max_pos};
    return launch_pdl(kern, dim3(G, c.H), dim3(kGenTile), sm, a.stream, static_cast<const T *>(a.q),
                      static_cast<const TC *>(c.S_K), static_cast<const TC *>(c.S_V),
                      static_cast<const TC *>(c.R_K), static_cast<const TC *>(c.R_V), a.page_table,
                      a.req_row, a.max_pages, c.num_pages, c.page_size, a.B, c.H, c.d_h, c.r,
                      scale_log2, sc, ws, a.status, static_cast<const T *>(a.B_K), rope,
                      static_cast<const T *>(c.N_K), cache_groups(c) * c.d_h, c.H / cache_groups(c));
}

template <typename T, typename TC>
static cudaError_t launch_split_generic_rp(const DecodeArgs &a, const DecodeWs &ws, int G) {
    if (!a.rope) return launch_split_generic_t<T, TC, 0>(a, ws, G);
    const int r = a.cache.r;  // the caller checks 1 <= r <= kRopeMaxRank
    if (r <= 16) return launch_split_generic_t<T, TC, 16>(a, ws, G);
    if (r <= 32) return launch_split_generic_t<T, TC, 32>(a, ws, G);
    if (r <= 48) return launch_split_generic_t<T, TC, 48>(a, ws, G);
    return launch_split_generic_t<T, TC, 64>(a, ws, G);
}

template <typename T>
cudaError_t launch_split_generic(const DecodeArgs &a, const DecodeWs &ws, int G) {
    if (a.cache.dtype == LRKV_FP8_E4M3) return launch_split_generic_rp<__nv_bfloat16, uint8_t>(a, ws, G);
    return launch_split_generic_rp<T, T>(a, ws, G);
}

// cos and sin of distance x theta_c, theta_c = base^(-2c/d_h), in double
// precision, rounded once to float and once (from the double) to f16.
__global__ void rope_table_kernel(double base, int d_h, int max_pos, float2 *table, __half2 *t16) {
    const int hc = d_h / 2;
    const size_t n = (size_t)max_pos * hc;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % hc);
        const double pos = (double)(i / hc);
        const double th = pow(base, -2.0 * c / d_h);
        double sv, cv;
        sincos(pos * th, &sv, &cv);
        table[i] = make_float2((float)cv, (float)sv);
        t16[i] = __halves2half2(__double2half(cv), __double2half(sv));
    }
}

cudaError_t launch_rope_table(double base, int d_h, int max_pos, void *table, cudaStream_t s) {
    const size_t n = (size_t)max_pos * (d_h / 2);
    const int blocks = (int)std::min<size_t>((n + 255) / 256, 4096);
    char *t = static_cast<char *>(table);
    rope_table_kernel<<<blocks, 256, 0, s>>>(base, d_h, max_pos, reinterpret_cast<float2 *>(t),
                                             reinterpret_cast<__half2 *>(t + rope_table_f16_offset(d_h, max_pos)));
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_combine(const DecodeArgs &a, const DecodeWs &ws, int G) {
    dim3 grid(a.cache.H, a.B);
    // d_h <= 256 columns of accS plus r <= 256 of accR: two columns per thread
    const bool staged = (size_t)a.cache.d_h * a.cache.r <= kStageFloats;
    const size_t bv_bytes = staged ? ((size_t)a.cache.d_h * a.cache.r * sizeof(T) + 15) / 16 * 16 : 0;
    const size_t sm = bv_bytes + sizeof(float) * ((size_t)a.cache.r + G);
    cudaError_t e = smem_limit_once(decode_combine_kernel<T>, 200 * 1024);
    if (e != cudaSuccess) return e;
    const int nthr = (a.cache.d_h + a.cache.r <= 256) ? 128 : 256;
    return launch_pdl(decode_combine_kernel<T>, grid, dim3(nthr), sm, a.stream,
                      static_cast<const T *>(a.B_V), a.B, a.cache.H, a.cache.d_h, a.cache.r,
                      staged, ws, static_cast<T *>(a.out));
}

template cudaError_t launch_prologue<float>(const DecodeArgs &, const DecodeWs &, int, int, bool);
template cudaError_t launch_prologue<__nv_bfloat16>(const DecodeArgs &, const DecodeWs &, int, int, bool);
template cudaError_t launch_split_generic<float>(const DecodeArgs &, const DecodeWs &, int);
template cudaError_t launch_split_generic<__nv_bfloat16>(const DecodeArgs &, const DecodeWs &, int);
template cudaError_t launch_combine<float>(const DecodeArgs &, const DecodeWs &, int);
template cudaError_t launch_combine<__nv_bfloat16>(const DecodeArgs &, const DecodeWs &, int);

}  // namespace lrkv
