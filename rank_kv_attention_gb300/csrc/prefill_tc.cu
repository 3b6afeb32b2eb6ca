// Causal LRKV prefill attention on 5th-generation tensor cores.
//
// "Low-Rank Key Value Attention", section 3, equations 6-7 applied to every
// query row of a prompt chunk: for request b, head h and query row i at
// position t_i, over the request's cached rows j <= t_i,
//   s_ij = (q_i . S_K[j] + (q_i B_K[h]) . R_K[h,j]) / sqrt(d_h)
//   o_i  = sum_j a_ij S_V[j] + (sum_j a_ij R_V[h,j]) B_V[h]^T,  a_i = softmax(s_i)
// (one softmax over both score branches, section 2).  The two score branches
// are one contraction over the concatenated width
//   [q | p_hi | p_lo] . [S_K | R_K[h] | R_K[h]]^T
// where p = q B_K[h] is split into two bf16 halves (p_hi + p_lo carries ~16
// mantissa bits), and the two value branches are one contraction
//   P . [S_V | R_V[h]]
// whose last r columns are expanded by B_V[h]^T once per query row at the end.
//
// One CTA = one (request, head, 128-row query tile), 6 warps:
//   warps 0-3  softmax and epilogue, thread = query row = tensor-memory lane;
//   warp 4     TMA producer (lane 0) and owner of the tensor-memory allocation;
//   warp 5     tcgen05.mma issuer (lane 0).
// Keys stream in tiles of 64 (one 64-row slice of a page; all four pools share
// the page id).  Tensor memory (512 columns): the [O_S | O_R] accumulator in
// columns 0..255, two 64-column score buffers at 256 and 320 (the score MMA of
// tile k+1 runs while the softmax of tile k reads the other buffer), p at 384;
// the final expansion reuses 256..383.  Softmax keeps a lazy running maximum
// (rescaling O in tensor memory only when the maximum grows by more than
// 2^8).  Keys past every row of the tile have their value rows cleared in
// shared memory, so whatever the cache holds there cannot reach the output.
#include <algorithm>

#include "append_kernels.cuh"
#include "tc_common.cuh"

namespace lrkv {

namespace {

constexpr int PF_BM = 128;                  // query rows per CTA
constexpr int PF_BN = 64;                   // keys per tile
constexpr int PF_CHUNK = PF_BM * 128;       // 128 rows x 128 bytes
constexpr int PF_BOX = PF_BN * 128;         // 64 rows x 128 bytes
constexpr int PF_KST = 2, PF_VST = 2;       // key / value ring stages
constexpr int PF_STAGE = 3 * PF_BOX;        // [S_*[:, 0:64] | S_*[:, 64:128] | R_*[h]]
constexpr int PF_OFF_QA = 0;                // q[0:64], q[64:128], p_hi, p_lo
constexpr int PF_OFF_PS = 4 * PF_CHUNK;     // two probability tiles [128 x 64]
constexpr int PF_OFF_K = PF_OFF_PS + 2 * PF_CHUNK;
constexpr int PF_OFF_V = PF_OFF_K + PF_KST * PF_STAGE;
constexpr int PF_OFF_BAR = PF_OFF_V + PF_VST * PF_STAGE;
constexpr uint32_t PF_TMEM_COLS = 512;
constexpr uint32_t PF_COL_S = 256, PF_COL_P = 384, PF_COL_E = 256;
constexpr float kPfLazyMax = 8.f;           // log2 units

struct PfBars {
    uint64_t q_full, pre_done, qa_ready, bv_full, ex_ready, ex_done, fin;
    uint64_t k_full[PF_KST], k_empty[PF_KST], v_full[PF_VST], v_empty[PF_VST];
    uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
    uint32_t tmem;
};
constexpr int PF_SMEM = PF_OFF_BAR + (int)sizeof(PfBars) + 1024;
static_assert(PF_SMEM <= 232448, "shared memory budget");

struct PfMaps {
    CUtensorMap q;       // Q [n, H, 128]: box 64 x 1 x 128
    CUtensorMap sk, sv;  // S_K, S_V pools [rows, 128]: box 64 x 64
    CUtensorMap rk, rv;  // R_K, R_V pools [rows, H r]: box 64 x 64
    CUtensorMap bk, bv;  // B_K, B_V [H 128, r]: box 64 x 64 (columns >= r read as 0)
};

struct PfArgs {
    const int32_t *cu_rows, *start_pos, *page_table;
    __nv_bfloat16 *out;
    int32_t *status;
    int n, B, H, r, page_size, max_pages, num_pages, max_len, n_qtiles;
    float scale_log2;  // log2(e) / sqrt(d_h)
};

__device__ __forceinline__ void st_shared16(uint8_t *p, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

// x -> (hi, lo) with hi = bf16(x), lo = bf16(x - hi), packed in pairs.
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - bf16lo(hi), x1 - bf16hi(hi));
}

template <int R16>
__global__ void __launch_bounds__(192, 1)
    prefill_tc_kernel(const __grid_constant__ PfMaps maps, const PfArgs a) {
    constexpr int NPV = 128 + 16 * R16;    // value columns [S_V | R_V[h] (padded)]
    constexpr int NO_LD = (NPV + 31) / 32; // 32-column groups of O
    extern __shared__ uint8_t pf_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(pf_smem_raw) + 1023) & ~uintptr_t(1023));
    PfBars &bar = *reinterpret_cast<PfBars *>(smem + PF_OFF_BAR);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, b = blockIdx.y, tq = a.n_qtiles - 1 - (int)blockIdx.z;

    if (tid == 0) {
        // single arrivals (TMA transaction counts, tcgen05.commit) ...
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.pre_done, 1);
        mbar_init(&bar.bv_full, 1);
        mbar_init(&bar.ex_done, 1);
        mbar_init(&bar.fin, 1);
        for (int k = 0; k < PF_KST; ++k) {
            mbar_init(&bar.k_full[k], 1);
            mbar_init(&bar.k_empty[k], 1);
        }
        for (int k = 0; k < PF_VST; ++k) {
            mbar_init(&bar.v_full[k], 1);
            mbar_init(&bar.v_empty[k], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&bar.s_full[k], 1);
            mbar_init(&bar.pv_done[k], 1);
            // ... and arrivals of all 128 softmax threads
            mbar_init(&bar.s_free[k], PF_BM);
            mbar_init(&bar.p_full[k], PF_BM);
        }
        mbar_init(&bar.qa_ready, PF_BM);
        mbar_init(&bar.ex_ready, PF_BM);
        fence_barrier_init();
    }
    if (tid == 128) {
        prefetch_tensormap(&maps.q);
        prefetch_tensormap(&maps.sk);
        prefetch_tensormap(&maps.sv);
        prefetch_tensormap(&maps.rk);
        prefetch_tensormap(&maps.rv);
    }
    pdl_wait();
    pdl_launch_dependents();

    // ---- tile geometry (identical in every thread)
    const int r0 = a.cu_rows[b], r1 = min(a.cu_rows[b + 1], a.n);
    if (r0 < 0 || r1 <= r0) return;
    const int i0 = r0 + tq * PF_BM;
    if (i0 >= r1) return;
    if (tq == a.n_qtiles - 1 && r1 > i0 + PF_BM) {  // rows beyond max_ctx: not covered
        if (tid == 0) status_or(a.status, LRKV_STATUS_BAD_SEQLEN);
    }
    const int nrows = min(PF_BM, r1 - i0);
    const int p0 = a.start_pos[b] + (i0 - r0);         // position of tile row 0
    const int t_lo = max(0, -p0), t_hi = min(nrows, a.max_len - p0);  // valid rows
    if (t_lo >= t_hi) {  // no row of this tile has a valid position: zero outputs
        if (tid < nrows) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((size_t)(i0 + tid) * a.H + h) * 128);
            for (int k = 0; k < 16; ++k) dst[k] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    const int max_p = p0 + t_hi - 1;
    const int nkt = max_p / PF_BN + 1;

    if (warp == 4) tmem_alloc(&bar.tmem, PF_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem;

    if (warp == 4) {
        if (lane == 0) {
            // ================= TMA producer =================
            bool ok = true;
            const int hr = h * a.r;
            mbar_arrive_expect_tx(&bar.q_full, 2 * PF_CHUNK + 2 * PF_BOX);
            tma_load_3d(smem + PF_OFF_QA, &maps.q, 0, h, i0, &bar.q_full);
            tma_load_3d(smem + PF_OFF_QA + PF_CHUNK, &maps.q, 64, h, i0, &bar.q_full);
            tma_load_2d(smem + PF_OFF_PS, &maps.bk, 0, h * 128, &bar.q_full);
            tma_load_2d(smem + PF_OFF_PS + PF_BOX, &maps.bk, 0, h * 128 + 64, &bar.q_full);
            int nk = 0, nv = 0;  // key / value tiles issued
            for (int kt = 0; kt < nkt; ++kt) {
                const int key0 = kt * PF_BN;
                const int32_t page = a.page_table[(size_t)b * a.max_pages + key0 / a.page_size];
                int y = -PF_BN;  // an invalid page reads as zeros (fully outside the pool)
                if (page < 0 || page >= a.num_pages) status_or(a.status, LRKV_STATUS_BAD_PAGE);
                else y = page * a.page_size + key0 % a.page_size;
                const int ks = kt % PF_KST, vs = kt % PF_VST;
                if (kt >= PF_KST && !mbar_wait(&bar.k_empty[ks], ((kt / PF_KST) - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *kb = smem + PF_OFF_K + ks * PF_STAGE;
                mbar_arrive_expect_tx(&bar.k_full[ks], PF_STAGE);
                tma_load_2d(kb, &maps.sk, 0, y, &bar.k_full[ks]);
                tma_load_2d(kb + PF_BOX, &maps.sk, 64, y, &bar.k_full[ks]);
                tma_load_2d(kb + 2 * PF_BOX, &maps.rk, hr, y, &bar.k_full[ks]);
                ++nk;
                if (kt >= PF_VST && !mbar_wait(&bar.v_empty[vs], ((kt / PF_VST) - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *vb = smem + PF_OFF_V + vs * PF_STAGE;
                mbar_arrive_expect_tx(&bar.v_full[vs], PF_STAGE);
                tma_load_2d(vb, &maps.sv, 0, y, &bar.v_full[vs]);
                tma_load_2d(vb + PF_BOX, &maps.sv, 64, y, &bar.v_full[vs]);
                tma_load_2d(vb + 2 * PF_BOX, &maps.rv, hr, y, &bar.v_full[vs]);
                ++nv;
            }
            // B_V[h] (K-major for the expansion) into the key stage tile nkt would use
            bool bv_issued = false;
            if (ok) {
                const int ks = nkt % PF_KST;
                if (nkt >= PF_KST && !mbar_wait(&bar.k_empty[ks], ((nkt / PF_KST) - 1) & 1)) {
                    ok = false;
                } else {
                    uint8_t *kb = smem + PF_OFF_K + ks * PF_STAGE;
                    mbar_arrive_expect_tx(&bar.bv_full, 2 * PF_BOX);
                    tma_load_2d(kb, &maps.bv, 0, h * 128, &bar.bv_full);
                    tma_load_2d(kb + PF_BOX, &maps.bv, 0, h * 128 + 64, &bar.bv_full);
                    bv_issued = true;
                }
            }
            if (!ok) status_or(a.status, LRKV_STATUS_TIMEOUT);
            // drain: every copy issued here has landed before the CTA can exit
            mbar_wait(&bar.q_full, 0);
            for (int s = 0; s < PF_KST && s < nk; ++s)
                mbar_wait(&bar.k_full[s], ((nk - 1 - s) / PF_KST) & 1);
            for (int s = 0; s < PF_VST && s < nv; ++s)
                mbar_wait(&bar.v_full[s], ((nv - 1 - s) / PF_VST) & 1);
            if (bv_issued) mbar_wait(&bar.bv_full, 0);
        }
    } else if (warp == 5) {
        if (lane == 0) {
            // ================= MMA issuer =================
            const uint32_t qa = smem_u32(smem + PF_OFF_QA), ps = smem_u32(smem + PF_OFF_PS);
            constexpr uint32_t id_s = tc_idesc_bf16(PF_BM, PF_BN);
            constexpr uint32_t id_pv = tc_idesc_bf16_bmn(PF_BM, NPV);
            constexpr uint32_t id_pre = tc_idesc_bf16_bmn(PF_BM, 64);
            constexpr uint32_t id_ex = tc_idesc_bf16(PF_BM, 128);
            bool ok = mbar_wait(&bar.q_full, 0);
            if (ok) {
                // p = q B_K[h]: A = q (K-major), B = B_K[h] rows (MN-major, one 64-column block)
                tc_fence_after();
                const uint64_t bkd = sw128_mnmajor_desc(ps, PF_BOX, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_f16(tmem + PF_COL_P, sw128_kmajor_desc(qa + (kk >> 2) * PF_CHUNK) + 2 * (kk & 3),
                               bkd + (uint64_t)(kk * 128), id_pre, kk != 0);
                tc_commit(&bar.pre_done);
                ok = mbar_wait(&bar.qa_ready, 0);
            }
            auto issue_scores = [&](int kt) -> bool {
                const int ks = kt % PF_KST;
                if (!mbar_wait(&bar.k_full[ks], (kt / PF_KST) & 1)) return false;
                if (kt >= 2 && !mbar_wait(&bar.s_free[kt & 1], ((kt - 2) >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + PF_OFF_K + ks * PF_STAGE);
                const uint32_t d = tmem + PF_COL_S + 64 * (kt & 1);
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_f16(d, sw128_kmajor_desc(qa + c * PF_CHUNK) + 2 * kk,
                                   sw128_kmajor_desc(kb + c * PF_BOX) + 2 * kk, id_s, (c | kk) != 0);
#pragma unroll
                for (int c = 2; c < 4; ++c)
#pragma unroll
                    for (int kk = 0; kk < R16; ++kk)
                        tc_mma_f16(d, sw128_kmajor_desc(qa + c * PF_CHUNK) + 2 * kk,
                                   sw128_kmajor_desc(kb + 2 * PF_BOX) + 2 * kk, id_s, 1);
                tc_commit(&bar.k_empty[ks]);
                tc_commit(&bar.s_full[kt & 1]);
                return true;
            };
            if (ok) ok = issue_scores(0);
            for (int kt = 0; kt < nkt && ok; ++kt) {
                if (kt + 1 < nkt && !(ok = issue_scores(kt + 1))) break;
                const int vs = kt % PF_VST;
                if (!mbar_wait(&bar.p_full[kt & 1], (kt >> 1) & 1) ||
                    !mbar_wait(&bar.v_full[vs], (kt / PF_VST) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sw128_kmajor_desc(ps + (kt & 1) * PF_CHUNK);
                const uint64_t vd =
                    sw128_mnmajor_desc(smem_u32(smem + PF_OFF_V + vs * PF_STAGE), PF_BOX, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // 16 keys per instruction
                    tc_mma_f16(tmem, ad + 2 * kk, vd + (uint64_t)(kk * 128), id_pv, (kt | kk) != 0);
                tc_commit(&bar.v_empty[vs]);
                tc_commit(&bar.pv_done[kt & 1]);
            }
            if (ok) ok = mbar_wait(&bar.ex_ready, 0) && mbar_wait(&bar.bv_full, 0);
            if (ok) {
                // E = (O_R / l)_hi B_V[h]^T + (O_R / l)_lo B_V[h]^T
                tc_fence_after();
                const uint32_t bvb = smem_u32(smem + PF_OFF_K + (nkt % PF_KST) * PF_STAGE);
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int kk = 0; kk < R16; ++kk)
                        tc_mma_f16(tmem + PF_COL_E, sw128_kmajor_desc(ps + c * PF_CHUNK) + 2 * kk,
                                   sw128_kmajor_desc(bvb) + 2 * kk, id_ex, (c | kk) != 0);
                tc_commit(&bar.ex_done);
            }
            if (!ok) status_or(a.status, LRKV_STATUS_TIMEOUT);
            tc_commit(&bar.fin);  // drain: all MMAs issued here are complete
            mbar_wait(&bar.fin, 0);
        }
    } else {
        // ================= softmax + epilogue: thread = query row =================
        const int t = tid;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const bool row_ok = t >= t_lo && t < t_hi;
        const int lim = row_ok ? p0 + t : -1;  // last visible key position
        float m = -INFINITY, l = 0.f;
        bool ok = __all_sync(0xffffffffu, mbar_wait(&bar.pre_done, 0));
        if (ok) {
            tc_fence_after();
            uint8_t *qh = smem + PF_OFF_QA + 2 * PF_CHUNK, *ql = qh + PF_CHUNK;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t v[32];
                tmem_ld32(lane_base + PF_COL_P + 32 * half, v);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        split_pack(__uint_as_float(v[8 * u + 2 * e]), __uint_as_float(v[8 * u + 2 * e + 1]),
                                   hi[e], lo[e]);
                    const uint32_t off = swz128(t, 4 * half + u);
                    st_shared16(qh + off, hi[0], hi[1], hi[2], hi[3]);
                    st_shared16(ql + off, lo[0], lo[1], lo[2], lo[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar.qa_ready);
        }
        for (int kt = 0; kt < nkt && ok; ++kt) {
            const int b2 = kt & 1, key0 = kt * PF_BN;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full[b2], (kt >> 1) & 1)))) break;
            tc_fence_after();
            float s[64];
            {
                uint32_t v[32];
                tmem_ld32(lane_base + PF_COL_S + 64 * b2, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(v[j]);
                tmem_ld32(lane_base + PF_COL_S + 64 * b2 + 32, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) s[32 + j] = __uint_as_float(v[j]);
            }
            tc_fence_before();
            mbar_arrive(&bar.s_free[b2]);
            const int32_t page = a.page_table[(size_t)b * a.max_pages + key0 / a.page_size];
            const int klim = (page >= 0 && page < a.num_pages) ? lim - key0 : -1;
            float mx = -INFINITY;
            if (klim >= PF_BN - 1) {
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    s[j] *= a.scale_log2;
                    mx = fmaxf(mx, s[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    s[j] = (j <= klim) ? s[j] * a.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, s[j]);
                }
            }
            const float m_new = (mx > m + kPfLazyMax) ? mx : m;
            const float alpha = (m_new == m) ? 1.f : exp2f(m - m_new);
            uint32_t pk[32];
            float sum = 0.f;
            if (m_new == -INFINITY) {
#pragma unroll
                for (int j = 0; j < 32; ++j) pk[j] = 0u;
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    pk[j] = pack_bf16(exp2f(s[2 * j] - m_new), exp2f(s[2 * j + 1] - m_new));
                    sum += bf16lo(pk[j]) + bf16hi(pk[j]);  // the weights the MMA sees
                }
            }
            l = l * alpha + sum;
            m = m_new;
            // probability buffer b2 is free once the value MMA of tile kt-2 is done
            if (kt >= 2 &&
                !(ok = __all_sync(0xffffffffu, mbar_wait(&bar.pv_done[b2], ((kt - 2) >> 1) & 1))))
                break;
            uint8_t *pb = smem + PF_OFF_PS + b2 * PF_CHUNK;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_shared16(pb + swz128(t, c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // the running maximum moved: rescale this row of O once the
                // value MMA of tile kt-1 has finished writing it
                const int pb1 = (kt - 1) & 1;
                if (!(ok = __all_sync(0xffffffffu,
                                      mbar_wait(&bar.pv_done[pb1], ((kt - 1) >> 1) & 1))))
                    break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < NO_LD; ++c) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + 32 * c, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
                    tmem_st32(lane_base + 32 * c, v);
                }
            }
            if (kt == nkt - 1 && max_p + 1 - key0 < PF_BN) {
                // keys past every row of this tile: clear their value rows
                const int vs = kt % PF_VST;
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.v_full[vs], (kt / PF_VST) & 1))))
                    break;
                const int z0 = max_p + 1 - key0, units = (PF_BN - z0) * 8;
                uint8_t *vb = smem + PF_OFF_V + vs * PF_STAGE + z0 * 128;
                for (int u = t; u < 3 * units; u += PF_BM) {
                    const int box = u / units, w = u - box * units;
                    st_shared16(vb + box * PF_BOX + w * 16, 0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar.p_full[b2]);
        }
        if (ok)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bar.pv_done[(nkt - 1) & 1], ((nkt - 1) >> 1) & 1));
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        if (ok) {
            // (O_R / l) split into bf16 halves, K-major, for the B_V[h] expansion
            tc_fence_after();
            uint8_t *eh = smem + PF_OFF_PS, *el = eh + PF_CHUNK;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t v[32];
                tmem_ld32(lane_base + 128 + 32 * half, v);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = 32 * half + 8 * u + 2 * e;
                        const float x0 = col < a.r ? __uint_as_float(v[8 * u + 2 * e]) * inv_l : 0.f;
                        const float x1 = col + 1 < a.r ? __uint_as_float(v[8 * u + 2 * e + 1]) * inv_l : 0.f;
                        split_pack(x0, x1, hi[e], lo[e]);
                    }
                    const uint32_t off = swz128(t, 4 * half + u);
                    st_shared16(eh + off, hi[0], hi[1], hi[2], hi[3]);
                    st_shared16(el + off, lo[0], lo[1], lo[2], lo[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar.ex_ready);
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.ex_done, 0));
        }
        if (ok) {
            tc_fence_after();
            __nv_bfloat16 *dst = a.out + ((size_t)(i0 + t) * a.H + h) * 128;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t vo[32], ve[32];
                tmem_ld32(lane_base + 32 * c, vo);
                tmem_ld32(lane_base + PF_COL_E + 32 * c, ve);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float y0 = __uint_as_float(vo[2 * e]) * inv_l + __uint_as_float(ve[2 * e]);
                    const float y1 = __uint_as_float(vo[2 * e + 1]) * inv_l + __uint_as_float(ve[2 * e + 1]);
                    pk[e] = row_ok ? pack_bf16(y0, y1) : 0u;
                }
                if (t < nrows) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
        } else if (lane == 0) {
            status_or(a.status, LRKV_STATUS_TIMEOUT);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, PF_TMEM_COLS);
    }
}

template <int R16>
cudaError_t launch_r16(const PfMaps &maps, const PfArgs &a, dim3 grid, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<R16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    return launch_pdl(prefill_tc_kernel<R16>, grid, dim3(192), PF_SMEM, s, maps, a);
}

}  // namespace

// Shape checks and tensor maps of one call; false when the shape is not covered.
static bool prefill_tc_plan(const PrefillTcArgs &p, PfMaps &maps, int &n_qtiles) {
    const lrkv_cache_t &c = p.cache;
    if (c.dtype != LRKV_BF16 || c.d_h != 128 || c.r < 8 || c.r > 64 || c.r % 8 != 0 ||
        c.page_size % PF_BN != 0 || c.H > 65535 || p.B > 65535 || p.n < 1 || p.max_ctx < 1)
        return false;
    const int64_t rows = (int64_t)c.num_pages * c.page_size;
    const int64_t max_len = (int64_t)p.max_pages * c.page_size;
    if (rows + PF_BN >= INT32_MAX || max_len >= INT32_MAX) return false;
    n_qtiles = (std::min(p.n, p.max_ctx) + PF_BM - 1) / PF_BM;
    if (n_qtiles > 65535) return false;
    const uint64_t Hr = (uint64_t)c.H * c.r;
    const uint64_t qdims[3] = {128, (uint64_t)c.H, (uint64_t)p.n};
    const uint64_t qstr[2] = {256, (uint64_t)c.H * 256};
    const uint32_t qbox[3] = {64, 1, PF_BM};
    const uint64_t kv_dims[2] = {128, (uint64_t)rows}, kv_str[1] = {256};
    const uint64_t r_dims[2] = {Hr, (uint64_t)rows}, r_str[1] = {Hr * 2};
    const uint64_t b_dims[2] = {(uint64_t)c.r, (uint64_t)c.H * 128}, b_str[1] = {(uint64_t)c.r * 2};
    const uint32_t box[2] = {64, 64};
    return tma_map_bf16(&maps.q, p.Q, 3, qdims, qstr, qbox) &&
           tma_map_bf16(&maps.sk, c.S_K, 2, kv_dims, kv_str, box) &&
           tma_map_bf16(&maps.sv, c.S_V, 2, kv_dims, kv_str, box) &&
           tma_map_bf16(&maps.rk, c.R_K, 2, r_dims, r_str, box) &&
           tma_map_bf16(&maps.rv, c.R_V, 2, r_dims, r_str, box) &&
           tma_map_bf16(&maps.bk, p.B_K, 2, b_dims, b_str, box) &&
           tma_map_bf16(&maps.bv, p.B_V, 2, b_dims, b_str, box);
}

bool prefill_tc_covers(const lrkv_cache_t &cache) {
    PrefillTcArgs p = {};
    p.cache = cache;
    p.Q = p.B_K = p.B_V = cache.S_K;  // any 16-byte aligned device address
    p.B = 1;
    p.n = 1;
    p.max_ctx = 1;
    p.max_pages = 1;
    PfMaps maps;
    int nq = 0;
    return prefill_tc_plan(p, maps, nq);
}

int launch_prefill_tc(const PrefillTcArgs &p) {
    const lrkv_cache_t &c = p.cache;
    PfMaps maps;
    int n_qtiles = 0;
    if (!prefill_tc_plan(p, maps, n_qtiles)) return 1;
    PfArgs a;
    a.cu_rows = p.cu_rows;
    a.start_pos = p.start_pos;
    a.page_table = p.page_table;
    a.out = static_cast<__nv_bfloat16 *>(p.out);
    a.status = p.status;
    a.n = p.n;
    a.B = p.B;
    a.H = c.H;
    a.r = c.r;
    a.page_size = c.page_size;
    a.max_pages = p.max_pages;
    a.num_pages = c.num_pages;
    a.max_len = p.max_pages * c.page_size;
    a.n_qtiles = n_qtiles;
    a.scale_log2 = 1.4426950408889634f / sqrtf(128.f);
    // heaviest query tiles (most keys) first: blockIdx.z counts tiles from the end
    const dim3 grid(c.H, p.B, n_qtiles);
    cudaError_t e;
    switch ((c.r + 15) / 16) {
        case 1: e = launch_r16<1>(maps, a, grid, p.stream); break;
        case 2: e = launch_r16<2>(maps, a, grid, p.stream); break;
        case 3: e = launch_r16<3>(maps, a, grid, p.stream); break;
        default: e = launch_r16<4>(maps, a, grid, p.stream); break;
    }
    return e == cudaSuccess ? 0 : -(int)e;
}

}  // namespace lrkv
