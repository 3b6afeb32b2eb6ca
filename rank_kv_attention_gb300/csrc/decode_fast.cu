// LRKV decode split kernel for bf16 caches with d_h = 128 (sm_103a).
//
// Reading note "Low-Rank Key Value Attention": section 3, Algorithm 2 and
// equations 6-7, fused as the note describes after Algorithm 2 (running max,
// exp-sum, a shared and a private value accumulator, both rescaled by the
// same factor when the max moves); section 4 on why the shared tile must be
// reused by all heads for the byte savings to show.
//
// One CTA streams a contiguous range of cache rows (possibly spanning
// several requests, see DecodePlan) for ALL H heads:
//   * a producer warp stages 16-row tiles into a ring of shared-memory stages:
//     S_K / S_V rows through 2-D TMA with 128-byte swizzle (read from HBM once
//     and reused by every head), and the tile's R_K / R_V rows (all heads
//     contiguous) through plain bulk copies; completion is tracked by
//     mbarriers;
//   * eight consumer warps score the tile: the shared part Q[H x 128] .
//     S_K^T[128 x 16] on tensor cores (mma.m16n8k16, bf16 in, fp32 acc), the
//     private part p_h . R_K[h, j] (rank r) with fp32 FMAs, one thread per
//     (head, row); one online softmax per head over the merged score; then
//     the shared value contraction P[H x 16] . S_V[16 x 128] on tensor cores
//     (P split into bf16 hi + lo so the weights keep ~16 mantissa bits) and
//     the private reduction a . R_V[h] with FMAs.
// Each (request, CTA) segment writes (m, l, accS, accR) to its partial slot;
// the combine kernel merges segments and expands accR by B_V^T once.
#include "decode_kernels.cuh"

namespace lrkv {

constexpr int cgcd(int a, int b) { return b == 0 ? a : cgcd(b, a % b); }

template <int H_, int R_, int STAGES_>
struct FastCfg {
    static constexpr int H = H_, R = R_, TS = 16, STAGES = STAGES_;
    static constexpr int DH = 128;
    static constexpr int NCW = 8, NC = NCW * 32, NT = NC;
    static constexpr int MT = H / 16;        // m16 tiles of heads
    static constexpr int NB = TS / 8;        // n8 blocks of rows in the score mma
    static constexpr int RC = R / 8;         // 16-byte chunks in one private row
    static constexpr int S_BOX = TS * 128;   // one 64-column half of a 16-row S tile
    static constexpr int S_BYTES = 2 * S_BOX;
    static constexpr int R_BYTES = TS * H * R * 2;
    static constexpr int OFF_SK = 0, OFF_SV = S_BYTES, OFF_RK = 2 * S_BYTES,
                         OFF_RV = 2 * S_BYTES + R_BYTES;
    static constexpr int STAGE = 2 * S_BYTES + 2 * R_BYTES;
    static constexpr int PAIRS = TS * H / NC;  // (row, head) pairs per thread per tile
    static constexpr int HPT = NC / H;         // threads sharing one head
    static constexpr int PST = TS + 8;         // padded row of the bf16 weight tile
    static constexpr int DISTINCT = 8 / cgcd(RC, 8);
    // shared-memory map after the stages
    static constexpr int OFF_BAR = STAGES * STAGE;
    static constexpr int OFF_SCS = OFF_BAR + 64;
    static constexpr int OFF_SCP = OFF_SCS + H * TS * 4;
    static constexpr int OFF_P32 = OFF_SCP + H * TS * 4;
    static constexpr int OFF_PB = OFF_P32 + H * TS * 4;
    static constexpr int OFF_M = OFF_PB + 2 * H * PST * 2;
    static constexpr int OFF_L = OFF_M + H * 4;
    static constexpr int OFF_A = OFF_L + H * 4;
    static constexpr int OFF_RED = OFF_A + H * 4;
    static constexpr int SMEM = OFF_RED + H * R * 4 + 1024;  // + alignment slack

    static_assert(H % 16 == 0 && NC % H == 0 && (TS * H) % NC == 0, "head mapping");
    static_assert(R % 8 == 0, "private rows are read in 16-byte chunks");
    static_assert(STAGE % 1024 == 0 && S_BOX % 1024 == 0, "128B-swizzle tiles need 1 KB alignment");
    static_assert(MT * NB <= NCW, "score tiles per warp");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct FastParams {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *R_K;
    const __nv_bfloat16 *R_V;
    const int32_t *page_table;
    const int32_t *req_row;
    int max_pages, num_pages, page_size, B;
    float scale_log2;
    DecodeWs ws;
    int32_t *status;
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Barrier over the 256 consumer threads that also ORs a flag across them.
__device__ __forceinline__ bool consumer_sync_or(bool v) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 q, %1, 0; barrier.cta.red.or.pred p, 1, 256, q; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ int find_request_fast(const int32_t *off, int B, int32_t x) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (off[mid + 1] > x) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16 *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}

// Walks the CTA's tile sequence (segments in order, 16-row tiles within a
// segment) ahead of the consumers and issues each tile's copies.  Only thread 0
// uses it.
template <class C>
struct TileIssuer {
    int b;
    int32_t start, end;
    int t, t_b;
    const int32_t *pt;
    bool done;

    __device__ void begin_segment(const FastParams &P) {
        while (P.ws.off[b + 1] <= start) ++b;
        const int32_t base = P.ws.off[b];
        const int32_t seg_end = min(end, P.ws.off[b + 1]);
        t = (start - base) / C::TS * C::TS;
        t_b = seg_end - base;
        pt = P.page_table + (size_t)(P.req_row ? P.req_row[b] : b) * P.max_pages;
    }

    __device__ void init(const FastParams &P, int b0, int32_t s0, int32_t e) {
        b = b0;
        start = s0;
        end = e;
        done = start >= end;
        if (!done) begin_segment(P);
    }

    // Issue the next tile into `stage`; returns false once the sequence is over.
    __device__ bool issue(const FastParams &P, const CUtensorMap *tmK, const CUtensorMap *tmV,
                          uint8_t *smem, uint64_t *full, int stage) {
        if (done) return false;
        int32_t page = pt[t / P.page_size];
        if (page < 0 || page >= P.num_pages) page = 0;  // consumers mask the tile
        const int row = page * P.page_size + t % P.page_size;
        uint8_t *st = smem + stage * C::STAGE;
        mbar_arrive_expect_tx(&full[stage], C::STAGE);
        tma_load_2d(st + C::OFF_SK, tmK, 0, row, &full[stage]);
        tma_load_2d(st + C::OFF_SK + C::S_BOX, tmK, 64, row, &full[stage]);
        tma_load_2d(st + C::OFF_SV, tmV, 0, row, &full[stage]);
        tma_load_2d(st + C::OFF_SV + C::S_BOX, tmV, 64, row, &full[stage]);
        const size_t roff = (size_t)row * C::H * C::R;
        bulk_load(st + C::OFF_RK, P.R_K + roff, C::R_BYTES, &full[stage]);
        bulk_load(st + C::OFF_RV, P.R_V + roff, C::R_BYTES, &full[stage]);
        t += C::TS;
        if (t >= t_b) {  // next segment
            start = P.ws.off[b] + t_b;
            if (start >= end) done = true;
            else begin_segment(P);
        }
        return true;
    }
};

template <class C>
__global__ void __launch_bounds__(C::NT, 1)
    decode_split_fast_kernel(const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const FastParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    float *sc_sh = reinterpret_cast<float *>(smem + C::OFF_SCS);
    float *sc_pr = reinterpret_cast<float *>(smem + C::OFF_SCP);
    float *p32 = reinterpret_cast<float *>(smem + C::OFF_P32);
    __nv_bfloat16 *pb = reinterpret_cast<__nv_bfloat16 *>(smem + C::OFF_PB);
    float *m_s = reinterpret_cast<float *>(smem + C::OFF_M);
    float *l_s = reinterpret_cast<float *>(smem + C::OFF_L);
    float *a_s = reinterpret_cast<float *>(smem + C::OFF_A);
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x;
    const DecodeWs &ws = P.ws;

    const int32_t total = ws.plan->total, chunk = ws.plan->chunk;
    const int32_t start0 = g * chunk;
    const int32_t end = min(total, start0 + chunk);
    if (start0 >= end) return;
    const int b0 = find_request_fast(ws.off, P.B, start0);

    // Thread 0 owns the barriers and the copy issue; it fills every stage up
    // front and then refills stage (k-1) % STAGES once the consumer barrier
    // after tile k's scores proves all warps are done with tile k-1.
    TileIssuer<C> issuer;
    uint32_t issued = 0;
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        issuer.init(P, b0, start0, end);
        for (int s = 0; s < C::STAGES; ++s)
            if (issuer.issue(P, &tmK, &tmV, smem, full, s)) ++issued;
    }
    __syncthreads();
    const int ps = P.page_size;

    // ------------------------------------------------------------------ consumers
    const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
    const int h_pr = tid % C::H;              // head of this thread's private work
    const int jj0 = tid / C::H;
    const int rot = ((tid & 7) / C::DISTINCT) % C::RC;  // bank-conflict-free chunk order
    const bool score_warp = warp < C::MT * C::NB;
    const int mt_s = warp / C::NB, nb_s = warp % C::NB;

    float p_rot[C::R];
    float accR[C::R];
    float accS[C::MT][2][4];
    uint32_t qf[8][4];

    uint32_t it = 0;
    int b = b0;
    int32_t start = start0;
    while (start < end) {
        while (ws.off[b + 1] <= start) ++b;
        const int32_t base = ws.off[b];
        const int32_t seg_end = min(end, ws.off[b + 1]);
        const int t_a = start - base, t_b = seg_end - base;
        const int32_t *pt = P.page_table + (size_t)(P.req_row ? P.req_row[b] : b) * P.max_pages;

        // -------- segment set-up
        if (tid < C::H) {
            m_s[tid] = -INFINITY;
            l_s[tid] = 0.f;
        }
        {
            const float *pp = ws.p + ((size_t)b * C::H + h_pr) * C::R;
#pragma unroll
            for (int c = 0; c < C::RC; ++c) {
                int ch = c + rot;
                if (ch >= C::RC) ch -= C::RC;
                const float4 v0 = *reinterpret_cast<const float4 *>(pp + ch * 8);
                const float4 v1 = *reinterpret_cast<const float4 *>(pp + ch * 8 + 4);
                p_rot[c * 8 + 0] = v0.x; p_rot[c * 8 + 1] = v0.y;
                p_rot[c * 8 + 2] = v0.z; p_rot[c * 8 + 3] = v0.w;
                p_rot[c * 8 + 4] = v1.x; p_rot[c * 8 + 5] = v1.y;
                p_rot[c * 8 + 6] = v1.z; p_rot[c * 8 + 7] = v1.w;
            }
        }
#pragma unroll
        for (int k = 0; k < C::R; ++k) accR[k] = 0.f;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) accS[mt][n][e] = 0.f;
        if (score_warp) {
            const __nv_bfloat16 *q0 = P.q + ((size_t)b * C::H + mt_s * 16 + gq) * C::DH + 2 * tq;
            const __nv_bfloat16 *q8 = q0 + 8 * C::DH;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qf[ks][0] = ld_u32(q0 + ks * 16);
                qf[ks][1] = ld_u32(q8 + ks * 16);
                qf[ks][2] = ld_u32(q0 + ks * 16 + 8);
                qf[ks][3] = ld_u32(q8 + ks * 16 + 8);
            }
        }

        // -------- stream the segment's tiles
        for (int t = t_a / C::TS * C::TS; t < t_b; t += C::TS, ++it) {
            const int s = it % C::STAGES;
            const bool got = mbar_wait(&full[s], (it / C::STAGES) & 1);
            const int32_t page = pt[t / ps];
            const bool page_ok = page >= 0 && page < P.num_pages;
            if (!page_ok && tid == 0) status_or(P.status, LRKV_STATUS_BAD_PAGE);
            const uint8_t *st = smem + s * C::STAGE;
            const bool partial = !page_ok || t < t_a || t + C::TS > t_b;

            if (got && partial) {
                // zero the S_V rows that are not visible so 0-weight x garbage
                // cannot reach the tensor-core accumulation
                const int row = tid >> 4, ch = tid & 15;
                const int tok = t + row;
                if (!(page_ok && tok >= t_a && tok < t_b)) {
                    uint8_t *dst = const_cast<uint8_t *>(st) + C::OFF_SV + (ch >> 3) * C::S_BOX +
                                   row * 128 + (ch & 7) * 16;
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();
                }
            }

            // A1: shared scores on tensor cores
            if (got && score_warp) {
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t skb = smem_u32(st + C::OFF_SK);
                const int mi = lane >> 3, rr = lane & 7;
                const int tok = nb_s * 8 + rr;
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                    const int ch = 4 * k2 + mi;
                    uint32_t b0r, b1r, b2r, b3r;
                    ldmatrix_x4(skb + (ch >> 3) * C::S_BOX + swz128(tok, ch & 7), b0r, b1r, b2r, b3r);
                    mma_bf16_16816(c, qf[2 * k2], b0r, b1r);
                    mma_bf16_16816(c, qf[2 * k2 + 1], b2r, b3r);
                }
                const int h0 = mt_s * 16 + gq, j0 = nb_s * 8 + 2 * tq;
                *reinterpret_cast<float2 *>(&sc_sh[h0 * C::TS + j0]) = make_float2(c[0], c[1]);
                *reinterpret_cast<float2 *>(&sc_sh[(h0 + 8) * C::TS + j0]) = make_float2(c[2], c[3]);
            }
            // A2: private scores p_h . R_K[h, j]
#pragma unroll
            for (int i = 0; i < C::PAIRS; ++i) {
                const int j = jj0 + i * C::HPT;
                const int tok = t + j;
                float acc = 0.f;
                if (got && page_ok && tok >= t_a && tok < t_b) {
                    const uint8_t *rk = st + C::OFF_RK + (j * C::H + h_pr) * (C::R * 2);
#pragma unroll
                    for (int c = 0; c < C::RC; ++c) {
                        int ch = c + rot;
                        if (ch >= C::RC) ch -= C::RC;
                        const uint4 v = *reinterpret_cast<const uint4 *>(rk + ch * 16);
                        acc = fmaf(p_rot[c * 8 + 0], bf16lo(v.x), acc);
                        acc = fmaf(p_rot[c * 8 + 1], bf16hi(v.x), acc);
                        acc = fmaf(p_rot[c * 8 + 2], bf16lo(v.y), acc);
                        acc = fmaf(p_rot[c * 8 + 3], bf16hi(v.y), acc);
                        acc = fmaf(p_rot[c * 8 + 4], bf16lo(v.z), acc);
                        acc = fmaf(p_rot[c * 8 + 5], bf16hi(v.z), acc);
                        acc = fmaf(p_rot[c * 8 + 6], bf16lo(v.w), acc);
                        acc = fmaf(p_rot[c * 8 + 7], bf16hi(v.w), acc);
                    }
                }
                sc_pr[h_pr * C::TS + j] = acc;
            }
            if (consumer_sync_or(!got)) {
                if (tid == 0) {
                    status_or(P.status, LRKV_STATUS_TIMEOUT);
                    // never leave with copies in flight into this CTA's shared memory
                    for (uint32_t k = it + 1; k < issued; ++k)
                        mbar_wait(&full[k % C::STAGES], (k / C::STAGES) & 1);
                }
                return;
            }
            // every warp has finished tile it-1: refill its stage
            if (tid == 0 && it > 0 && issuer.issue(P, &tmK, &tmV, smem, full, (it - 1) % C::STAGES))
                ++issued;

            // B: merged score, online softmax per head (16 lanes per head)
#pragma unroll
            for (int i = 0; i < C::PAIRS; ++i) {
                const int e = tid + i * C::NC;
                const int h = e / C::TS, j = e % C::TS;
                const int tok = t + j;
                const bool v = page_ok && tok >= t_a && tok < t_b;
                const float sv = v ? (sc_sh[h * C::TS + j] + sc_pr[h * C::TS + j]) * P.scale_log2
                                   : -INFINITY;
                float mx = sv;
#pragma unroll
                for (int o = C::TS / 2; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_old = m_s[h];
                const float m_new = fmaxf(m_old, mx);
                float alpha = 1.f, pe = 0.f;
                if (m_new != -INFINITY) {
                    alpha = exp2f(m_old - m_new);
                    pe = v ? exp2f(sv - m_new) : 0.f;
                }
                float sum = pe;
#pragma unroll
                for (int o = C::TS / 2; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                p32[h * C::TS + j] = pe;
                const __nv_bfloat16 hi = __float2bfloat16_rn(pe);
                const __nv_bfloat16 lo = __float2bfloat16_rn(pe - __bfloat162float(hi));
                pb[h * C::PST + j] = hi;
                pb[C::H * C::PST + h * C::PST + j] = lo;
                if (j == 0) {
                    m_s[h] = m_new;
                    l_s[h] = l_s[h] * alpha + sum;
                    a_s[h] = alpha;
                }
            }
            consumer_sync();

            // C1: shared value accumulation on tensor cores
            {
                const uint32_t svb = smem_u32(st + C::OFF_SV);
                const int mi = lane >> 3, rr = lane & 7;
                const int tok = (mi & 1) * 8 + rr;
                const int ch = 2 * warp + (mi >> 1);
                uint32_t b00, b01, b10, b11;
                ldmatrix_x4_trans(svb + (ch >> 3) * C::S_BOX + swz128(tok, ch & 7), b00, b01, b10, b11);
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    const int h0 = mt * 16 + gq;
                    const float al0 = a_s[h0], al8 = a_s[h0 + 8];
#pragma unroll
                    for (int n = 0; n < 2; ++n) {
                        accS[mt][n][0] *= al0; accS[mt][n][1] *= al0;
                        accS[mt][n][2] *= al8; accS[mt][n][3] *= al8;
                    }
                    uint32_t ah[4], alw[4];
                    const __nv_bfloat16 *ph = pb + h0 * C::PST + 2 * tq;
                    const __nv_bfloat16 *pl = ph + C::H * C::PST;
                    ah[0] = ld_u32(ph);                 ah[1] = ld_u32(ph + 8 * C::PST);
                    ah[2] = ld_u32(ph + 8);             ah[3] = ld_u32(ph + 8 * C::PST + 8);
                    alw[0] = ld_u32(pl);                alw[1] = ld_u32(pl + 8 * C::PST);
                    alw[2] = ld_u32(pl + 8);            alw[3] = ld_u32(pl + 8 * C::PST + 8);
                    mma_bf16_16816(accS[mt][0], ah, b00, b01);
                    mma_bf16_16816(accS[mt][0], alw, b00, b01);
                    mma_bf16_16816(accS[mt][1], ah, b10, b11);
                    mma_bf16_16816(accS[mt][1], alw, b10, b11);
                }
            }
            // C2: private value accumulation a . R_V[h]
            {
                const float al = a_s[h_pr];
#pragma unroll
                for (int k = 0; k < C::R; ++k) accR[k] *= al;
#pragma unroll
                for (int i = 0; i < C::PAIRS; ++i) {
                    const int j = jj0 + i * C::HPT;
                    const int tok = t + j;
                    if (page_ok && tok >= t_a && tok < t_b) {
                        const float pj = p32[h_pr * C::TS + j];
                        const uint8_t *rv = st + C::OFF_RV + (j * C::H + h_pr) * (C::R * 2);
#pragma unroll
                        for (int c = 0; c < C::RC; ++c) {
                            int ch = c + rot;
                            if (ch >= C::RC) ch -= C::RC;
                            const uint4 v = *reinterpret_cast<const uint4 *>(rv + ch * 16);
                            accR[c * 8 + 0] = fmaf(pj, bf16lo(v.x), accR[c * 8 + 0]);
                            accR[c * 8 + 1] = fmaf(pj, bf16hi(v.x), accR[c * 8 + 1]);
                            accR[c * 8 + 2] = fmaf(pj, bf16lo(v.y), accR[c * 8 + 2]);
                            accR[c * 8 + 3] = fmaf(pj, bf16hi(v.y), accR[c * 8 + 3]);
                            accR[c * 8 + 4] = fmaf(pj, bf16lo(v.z), accR[c * 8 + 4]);
                            accR[c * 8 + 5] = fmaf(pj, bf16hi(v.z), accR[c * 8 + 5]);
                            accR[c * 8 + 6] = fmaf(pj, bf16lo(v.w), accR[c * 8 + 6]);
                            accR[c * 8 + 7] = fmaf(pj, bf16hi(v.w), accR[c * 8 + 7]);
                        }
                    }
                }
            }
        }

        // -------- segment end: write the partial state of slot b + g
        consumer_sync();
        const size_t slot = (size_t)b + g;
        const size_t W = C::DH + C::R;
        if (tid < C::H) {
            ws.ml[(slot * C::H + tid) * 2 + 0] = m_s[tid];
            ws.ml[(slot * C::H + tid) * 2 + 1] = l_s[tid];
        }
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int h0 = mt * 16 + gq;
                const int d = 16 * warp + 8 * n + 2 * tq;
                *reinterpret_cast<float2 *>(&ws.acc[(slot * C::H + h0) * W + d]) =
                    make_float2(accS[mt][n][0], accS[mt][n][1]);
                *reinterpret_cast<float2 *>(&ws.acc[(slot * C::H + h0 + 8) * W + d]) =
                    make_float2(accS[mt][n][2], accS[mt][n][3]);
            }
        // private accumulators: threads sharing a head are summed in a fixed order
        if (C::H == 16) {
#pragma unroll
            for (int k = 0; k < C::R; ++k) accR[k] += __shfl_xor_sync(0xffffffffu, accR[k], 16);
        }
        for (int w = 0; w < C::NCW; ++w) {
            if (warp == w && lane < C::H) {
#pragma unroll
                for (int c = 0; c < C::RC; ++c) {
                    int ch = c + rot;
                    if (ch >= C::RC) ch -= C::RC;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float *dst = &red[h_pr * C::R + ch * 8 + e];
                        *dst = (w == 0) ? accR[c * 8 + e] : *dst + accR[c * 8 + e];
                    }
                }
            }
            consumer_sync();
        }
        for (int i = tid; i < C::H * C::R; i += C::NC) {
            const int h = i / C::R, k = i % C::R;
            ws.acc[(slot * C::H + h) * W + C::DH + k] = red[i];
        }
        consumer_sync();
        start = seg_end;
    }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and dispatch
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D map over an S pool viewed as [rows, 128] bf16; box = 16 rows x 64 columns,
// 128-byte swizzle (matches swz128 on the device side).
static bool make_s_map(CUtensorMap *map, const void *pool, int64_t rows) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    cuuint64_t strides[1] = {128 * 2};
    cuuint32_t box[2] = {64, 16};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int H, int R>
struct Pick {
    static constexpr int stage = FastCfg<H, R, 1>::STAGE;
    static constexpr int misc = FastCfg<H, R, 1>::SMEM - FastCfg<H, R, 1>::OFF_BAR;
    static constexpr int fit = (227 * 1024 - misc) / stage;
    static constexpr int STAGES = fit > 4 ? 4 : fit;
    using Cfg = FastCfg<H, R, STAGES>;
};

template <int H, int R>
static cudaError_t launch_fast_cfg(const DecodeArgs &a, const DecodeWs &ws, int G) {
    using C = typename Pick<H, R>::Cfg;
    static_assert(Pick<H, R>::STAGES >= 2, "at least double buffering");
    const auto &c = a.cache;
    CUtensorMap mk, mv;
    const int64_t rows = (int64_t)c.num_pages * c.page_size;
    if (!make_s_map(&mk, c.S_K, rows) || !make_s_map(&mv, c.S_V, rows))
        return cudaErrorInvalidValue;
    auto kern = decode_split_fast_kernel<C>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    FastParams P;
    P.q = static_cast<const __nv_bfloat16 *>(a.q);
    P.R_K = static_cast<const __nv_bfloat16 *>(c.R_K);
    P.R_V = static_cast<const __nv_bfloat16 *>(c.R_V);
    P.page_table = a.page_table;
    P.req_row = a.req_row;
    P.max_pages = a.max_pages;
    P.num_pages = c.num_pages;
    P.page_size = c.page_size;
    P.B = a.B;
    P.scale_log2 = 1.4426950408889634f / sqrtf(128.f);
    P.ws = ws;
    P.status = a.status;
    kern<<<G, C::NT, C::SMEM, a.stream>>>(mk, mv, P);
    return cudaGetLastError();
}

#define LRKV_FAST_SHAPES(X) X(16, 16) X(16, 32) X(16, 48) X(16, 56) X(16, 64) X(32, 16) X(32, 32)

bool fast_decode_supported(int H, int d_h, int r, int page_size, int dtype) {
    if (dtype != LRKV_BF16 || d_h != 128 || page_size % 16 != 0) return false;
    if (!get_encode_tiled()) return false;
#define X(h, rr) if (H == h && r == rr) return true;
    LRKV_FAST_SHAPES(X)
#undef X
    return false;
}

int fast_decode_grid(int, int) { return device_sm_count(); }

cudaError_t launch_split_fast(const DecodeArgs &a, const DecodeWs &ws, int G) {
    const int H = a.cache.H, r = a.cache.r;
#define X(h, rr) if (H == h && r == rr) return launch_fast_cfg<h, rr>(a, ws, G);
    LRKV_FAST_SHAPES(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace lrkv
