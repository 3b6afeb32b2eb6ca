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
// One CTA = one (request, head) and two adjacent 128-row query tiles A and B
// that share every key/value tile, 10 warps:
//   warps 0-3  softmax + epilogue of tile A, thread = query row = TMEM lane;
//   warps 4-7  the same for tile B;
//   warp 8     TMA producer (lane 0), owner of the tensor-memory allocation;
//   warp 9     tcgen05.mma issuer (lane 0).
// The issuer alternates between the tiles (P.V of A, scores of A's next key
// tile, P.V of B, scores of B's next), so the tensor core works on one tile
// while the other tile's softmax runs.  Keys stream in tiles of 64 (one
// 64-row slice of a page; all four pools share the page id).
//
// Tensor memory (512 columns): tile T owns columns [256 T, 256 T + 256):
// the [O_S | O_R] accumulator in 0..191, the 64 fp32 scores in 192..255, which
// the softmax overwrites with the bf16 probabilities (columns 192..223) that
// the value MMA reads as its A operand.  p = q B_K[h] lands in the score
// columns before the loop; the final expansion uses 128..255.  tcgen05.mma
// runs in issue order, so the scores of key tile k+1 (issued after the value
// MMA of tile k) never overwrite probabilities still being read.
//
// Softmax keeps a lazy running maximum (O is rescaled in tensor memory only
// when the maximum grows by more than 2^8).  Keys past every row of the CTA
// have their value rows cleared in shared memory, so whatever the cache holds
// there cannot reach the output.
#include <algorithm>

#include "append_kernels.cuh"
#include "tc_common.cuh"

namespace lrkv {

namespace {

constexpr int PF_BM = 128;                  // query rows per tile (two tiles per CTA)
constexpr int PF_BN = 64;                   // keys per tile
constexpr int PF_CHUNK = PF_BM * 128;       // 128 rows x 128 bytes
constexpr int PF_BOX = PF_BN * 128;         // 64 rows x 128 bytes
constexpr int PF_KST = 2, PF_VST = 2;       // key / value ring stages
constexpr int PF_STAGE = 3 * PF_BOX;        // [S_*[:, 0:64] | S_*[:, 64:128] | R_*[h]]
constexpr int PF_QA = 4 * PF_CHUNK;         // per tile: q[0:64], q[64:128], p_hi, p_lo
constexpr int PF_OFF_K = 2 * PF_QA;
constexpr int PF_OFF_V = PF_OFF_K + PF_KST * PF_STAGE;
constexpr int PF_OFF_BAR = PF_OFF_V + PF_VST * PF_STAGE;
constexpr int PF_OFF_BK = PF_QA + 2 * PF_CHUNK;  // B_K[h] staged in tile B's p_hi chunk
constexpr int PF_THREADS = 320;
constexpr uint32_t PF_TMEM_COLS = 512;
constexpr uint32_t PF_COL_S = 192, PF_COL_E = 128;  // within a tile's 256 columns
constexpr float kPfLazyMax = 8.f;                    // log2 units

struct PfBars {
    uint64_t q_full, pre_done, bv_full, fin;
    uint64_t k_full[PF_KST], k_empty[PF_KST], v_full[PF_VST], v_empty[PF_VST];
    uint64_t qa_ready[2], s_full[2], p_full[2], pv_done[2], ex_ready[2], ex_done[2];
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
    int n, B, H, r, page_size, max_pages, num_pages, max_len, n_pairs;
    float scale_log2;  // log2(e) / sqrt(d_h)
};

__device__ __forceinline__ void st_shared16(uint8_t *p, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

// 2^x on the special-function unit (PTX ex2.approx.ftz: ~2 ulp; -inf -> +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// x -> (hi, lo) with hi = bf16(x), lo = bf16(x - hi), packed in pairs.
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - bf16lo(hi), x1 - bf16hi(hi));
}

// Rows of one 128-row query tile.
struct PfTile {
    int row0;    // first global row
    int nrows;   // rows of the request in this tile (0..128)
    int p0;      // position of tile row 0
    int t_lo, t_hi;  // rows with a valid position: [t_lo, t_hi)
    int nkt;     // key tiles this tile attends to (0: none)
    int max_p;   // last visible key position (valid when nkt > 0)
};

__device__ __forceinline__ PfTile pf_tile(int row0, int r0, int r1, int start, int max_len) {
    PfTile t;
    t.row0 = row0;
    t.nrows = max(0, min(PF_BM, r1 - row0));
    t.p0 = start + (row0 - r0);
    t.t_lo = max(0, -t.p0);
    t.t_hi = min(t.nrows, max_len - t.p0);
    if (t.t_lo < t.t_hi) {
        t.max_p = t.p0 + t.t_hi - 1;
        t.nkt = t.max_p / PF_BN + 1;
    } else {
        t.max_p = -1;
        t.nkt = 0;
    }
    return t;
}

// Scores of one key tile: [q | p_hi | p_lo] . [S_K | R_K[h] | R_K[h]]^T into
// 64 fp32 columns at d.  q[c]: lower descriptor words of the tile's four A
// chunks; k[c]: of the key stage's three boxes.
template <int R16>
__device__ __forceinline__ void issue_scores(uint32_t d, const uint32_t (&q)[4], const uint32_t (&k)[3]) {
    constexpr uint32_t id_s = tc_idesc_bf16(PF_BM, PF_BN);
#pragma unroll
    for (int c = 0; c < 2; ++c)  // q . S_K
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) tc_mma_lo(d, q[c] + 2 * kk, k[c] + 2 * kk, id_s, (c | kk) != 0);
#pragma unroll
    for (int c = 2; c < 4; ++c)  // p_hi . R_K[h] + p_lo . R_K[h]
#pragma unroll
        for (int kk = 0; kk < R16; ++kk) tc_mma_lo(d, q[c] + 2 * kk, k[2] + 2 * kk, id_s, 1);
}

// Packed pairs of fp32 (PTX f32x2 arithmetic, sm_100 family).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

template <int R16>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ PfMaps maps, const PfArgs a) {
    constexpr int NPV = 128 + 16 * R16;    // value columns [S_V | R_V[h] (padded)]
    constexpr int NO_LD = (NPV + 31) / 32; // 32-column groups of O
    extern __shared__ uint8_t pf_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(pf_smem_raw) + 1023) & ~uintptr_t(1023));
    PfBars &bar = *reinterpret_cast<PfBars *>(smem + PF_OFF_BAR);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, b = blockIdx.y, tp = a.n_pairs - 1 - (int)blockIdx.z;

    if (tid == 0) {
        // single arrivals (TMA transaction counts, tcgen05.commit) ...
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.pre_done, 1);
        mbar_init(&bar.bv_full, 1);
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
            mbar_init(&bar.ex_done[k], 1);
            // ... and arrivals of a tile's 128 softmax threads
            mbar_init(&bar.qa_ready[k], PF_BM);
            mbar_init(&bar.p_full[k], PF_BM);
            mbar_init(&bar.ex_ready[k], PF_BM);
        }
        fence_barrier_init();
    }
    if (tid == 256) {
        prefetch_tensormap(&maps.q);
        prefetch_tensormap(&maps.sk);
        prefetch_tensormap(&maps.sv);
        prefetch_tensormap(&maps.rk);
        prefetch_tensormap(&maps.rv);
    }
    pdl_wait();
    pdl_launch_dependents();

    // ---- geometry (identical in every thread)
    const int r0 = a.cu_rows[b], r1 = min(a.cu_rows[b + 1], a.n);
    if (r0 < 0 || r1 <= r0) return;
    const int i0 = r0 + tp * 2 * PF_BM;
    if (i0 >= r1) return;
    if (tp == a.n_pairs - 1 && r1 > i0 + 2 * PF_BM) {  // rows beyond max_ctx: not covered
        if (tid == 0) status_or(a.status, LRKV_STATUS_BAD_SEQLEN);
    }
    const int start = a.start_pos[b];
    const PfTile tl[2] = {pf_tile(i0, r0, r1, start, a.max_len),
                          pf_tile(i0 + PF_BM, r0, r1, start, a.max_len)};
    const int nkt0 = tl[0].nkt, nkt1 = tl[1].nkt;  // key tiles of tiles A and B
    const int nkt = max(nkt0, nkt1);
    const int max_p = max(tl[0].max_p, tl[1].max_p);  // last key any row of the CTA sees
    if (nkt == 0) {  // no row has a valid position: zero outputs
        if (tid < 2 * PF_BM && (tid & 127) < (tid >> 7 ? tl[1].nrows : tl[0].nrows)) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((size_t)(i0 + tid) * a.H + h) * 128);
            for (int k = 0; k < 16; ++k) dst[k] = make_uint4(0, 0, 0, 0);
        }
        return;
    }

    if (warp == 8) tmem_alloc(&bar.tmem, PF_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem;

    if (warp == 8) {
        if (lane == 0) {
            // ================= TMA producer =================
            bool ok = true;
            const int hr = h * a.r;
            uint32_t tx = 2 * PF_BOX;
            tx += (nkt0 ? 2 * PF_CHUNK : 0) + (nkt1 ? 2 * PF_CHUNK : 0);
            mbar_arrive_expect_tx(&bar.q_full, tx);
            for (int T = 0; T < 2; ++T) {
                if (!(T ? nkt1 : nkt0)) continue;
                tma_load_3d(smem + T * PF_QA, &maps.q, 0, h, i0 + T * PF_BM, &bar.q_full);
                tma_load_3d(smem + T * PF_QA + PF_CHUNK, &maps.q, 64, h, i0 + T * PF_BM, &bar.q_full);
            }
            tma_load_2d(smem + PF_OFF_BK, &maps.bk, 0, h * 128, &bar.q_full);
            tma_load_2d(smem + PF_OFF_BK + PF_BOX, &maps.bk, 0, h * 128 + 64, &bar.q_full);
            int nk = 0, nv = 0;  // key / value tiles issued
            for (int kt = 0; kt < nkt; ++kt) {
                const int key0 = kt * PF_BN;
                const int32_t page = a.page_table[(size_t)b * a.max_pages + key0 / a.page_size];
                int y = -PF_BN;  // an invalid page reads as zeros (fully outside the pool)
                if (page < 0 || page >= a.num_pages) status_or(a.status, LRKV_STATUS_BAD_PAGE);
                else y = page * a.page_size + key0 % a.page_size;
                const int ks = kt % PF_KST, vs = kt % PF_VST;
                if (kt >= PF_KST && !mbar_wait_sleep(&bar.k_empty[ks], ((kt / PF_KST) - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *kb = smem + PF_OFF_K + ks * PF_STAGE;
                mbar_arrive_expect_tx(&bar.k_full[ks], PF_STAGE);
                tma_load_2d(kb, &maps.sk, 0, y, &bar.k_full[ks]);
                tma_load_2d(kb + PF_BOX, &maps.sk, 64, y, &bar.k_full[ks]);
                tma_load_2d(kb + 2 * PF_BOX, &maps.rk, hr, y, &bar.k_full[ks]);
                ++nk;
                if (kt >= PF_VST && !mbar_wait_sleep(&bar.v_empty[vs], ((kt / PF_VST) - 1) & 1)) {
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
                if (nkt >= PF_KST && !mbar_wait_sleep(&bar.k_empty[ks], ((nkt / PF_KST) - 1) & 1)) {
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
            mbar_wait_sleep(&bar.q_full, 0);
            for (int s = 0; s < PF_KST && s < nk; ++s)
                mbar_wait_sleep(&bar.k_full[s], ((nk - 1 - s) / PF_KST) & 1);
            for (int s = 0; s < PF_VST && s < nv; ++s)
                mbar_wait_sleep(&bar.v_full[s], ((nv - 1 - s) / PF_VST) & 1);
            if (bv_issued) mbar_wait_sleep(&bar.bv_full, 0);
        }
    } else if (warp == 9) {
        if (lane == 0) {
            // ================= MMA issuer =================
            static_assert(PF_KST == 2 && PF_VST == 2, "stage parities below assume two stages");
            constexpr uint32_t id_pv = tc_idesc_bf16_bmn(PF_BM, NPV);
            constexpr uint32_t id_pre = tc_idesc_bf16_bmn(PF_BM, 64);
            const uint32_t qa0 = smem_u32(smem);
            // lower descriptor words: tile T's four A chunks, each stage's key boxes and value block
            uint32_t qlo[2][4], klo[2][3], vlo[2];
#pragma unroll
            for (int T = 0; T < 2; ++T)
#pragma unroll
                for (int c = 0; c < 4; ++c) qlo[T][c] = sw128_desc_lo(qa0 + T * PF_QA + c * PF_CHUNK, 16);
#pragma unroll
            for (int st = 0; st < 2; ++st) {
#pragma unroll
                for (int c = 0; c < 3; ++c)
                    klo[st][c] = sw128_desc_lo(qa0 + PF_OFF_K + st * PF_STAGE + c * PF_BOX, 16);
                vlo[st] = sw128_desc_lo(qa0 + PF_OFF_V + st * PF_STAGE, PF_BOX);
            }
            bool ok = mbar_wait_sleep(&bar.q_full, 0);
            if (ok) {
                // p = q B_K[h]: A = q (K-major), B = B_K[h] rows (MN-major, one 64-column block)
                tc_fence_after();
                const uint32_t bk = sw128_desc_lo(qa0 + PF_OFF_BK, PF_BOX);
#pragma unroll
                for (int T = 0; T < 2; ++T) {
                    if (!(T ? nkt1 : nkt0)) continue;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc_mma_lo(tmem + 256 * T + PF_COL_S, qlo[T][kk >> 2] + 2 * (kk & 3), bk + 128 * kk,
                                  id_pre, kk != 0);
                }
                tc_commit(&bar.pre_done);
                for (int T = 0; T < 2 && ok; ++T)
                    if (T ? nkt1 : nkt0) ok = mbar_wait_sleep(&bar.qa_ready[T], 0);
            }
            // Key tile kt is used by tile T iff kt < nkt_T; tile B (positions
            // after A's) is its last user whenever it uses it.
            // Scores of key tile 0.
            if (ok) ok = mbar_wait_sleep(&bar.k_full[0], 0);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int T = 0; T < 2; ++T) {
                    if (!(T ? nkt1 : nkt0)) continue;
                    issue_scores<R16>(tmem + 256 * T + PF_COL_S, qlo[T], klo[0]);
                    tc_commit(&bar.s_full[T]);
                }
                tc_commit(&bar.k_empty[0]);
            }
            // One group per (key tile, query tile): wait for everything first,
            // then P.V of tile kt and the scores of tile kt+1 back to back.
            for (int kt = 0; kt < nkt && ok; ++kt) {
#pragma unroll
                for (int T = 0; T < 2; ++T) {
                    const int nkt_t = T ? nkt1 : nkt0;
                    if (kt >= nkt_t || !ok) continue;
                    const int vs = kt & 1, ks = (kt + 1) & 1;
                    const bool v_first = T == 0 || kt >= nkt0, v_last = T == 1 || kt >= nkt1;
                    const bool more = kt + 1 < nkt_t;
                    const bool k_first = T == 0 || kt + 1 >= nkt0, k_last = T == 1 || kt + 1 >= nkt1;
                    if (!mbar_wait_sleep(&bar.p_full[T], kt & 1) ||
                        (v_first && !mbar_wait_sleep(&bar.v_full[vs], (kt >> 1) & 1)) ||
                        (more && k_first && !mbar_wait_sleep(&bar.k_full[ks], ((kt + 1) >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t vb = vs ? vlo[1] : vlo[0];
                    const uint32_t pa = tmem + 256 * T + PF_COL_S;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // 16 keys (8 packed columns) per instruction
                        tc_mma_ts_lo(tmem + 256 * T, pa + 8 * kk, vb + 128 * kk, id_pv, (kt | kk) != 0);
                    tc_commit(&bar.pv_done[T]);
                    if (v_last) tc_commit(&bar.v_empty[vs]);
                    if (more) {
                        issue_scores<R16>(tmem + 256 * T + PF_COL_S, qlo[T], ks ? klo[1] : klo[0]);
                        tc_commit(&bar.s_full[T]);
                        if (k_last) tc_commit(&bar.k_empty[ks]);
                    }
                }
            }
            // E_T = (O_R / l)_hi B_V[h]^T + (O_R / l)_lo B_V[h]^T into columns 128..255
            constexpr uint32_t id_ex = tc_idesc_bf16(PF_BM, 128);
            const uint32_t bvb = smem_u32(smem + PF_OFF_K + (nkt % PF_KST) * PF_STAGE);
            bool bv_ready = false;
            for (int T = 0; T < 2 && ok; ++T) {
                if (!(T ? nkt1 : nkt0)) continue;
                if (!mbar_wait_sleep(&bar.ex_ready[T], 0) || (!bv_ready && !mbar_wait_sleep(&bar.bv_full, 0))) {
                    ok = false;
                    break;
                }
                bv_ready = true;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int kk = 0; kk < R16; ++kk)
                        tc_mma_f16(tmem + 256 * T + PF_COL_E,
                                   sw128_kmajor_desc(qa0 + T * PF_QA + c * PF_CHUNK) + 2 * kk,
                                   sw128_kmajor_desc(bvb) + 2 * kk, id_ex, (c | kk) != 0);
                tc_commit(&bar.ex_done[T]);
            }
            if (!ok) status_or(a.status, LRKV_STATUS_TIMEOUT);
            tc_commit(&bar.fin);  // drain: all MMAs issued here are complete
            mbar_wait_sleep(&bar.fin, 0);
        }
    } else {
        // ================= softmax + epilogue: thread = query row of tile T =================
        const int T = warp >> 2, t = tid & 127;
        const PfTile tt = T ? tl[1] : tl[0];
        const uint32_t lane_base = tmem + 256 * T + ((uint32_t)((warp & 3) * 32) << 16);
        uint8_t *qa = smem + T * PF_QA;
        const bool row_ok = t >= tt.t_lo && t < tt.t_hi;
        __nv_bfloat16 *dst = a.out + ((size_t)(tt.row0 + t) * a.H + h) * 128;
        if (!tt.nkt) {
            if (t < tt.nrows) {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
                for (int k = 0; k < 16; ++k) d4[k] = make_uint4(0, 0, 0, 0);
            }
        } else {
            const int lim = row_ok ? tt.p0 + t : -1;  // last visible key position
            // the first tile to use the last key tile clears its value rows past max_p
            const bool clears = (T == 0) == (nkt - 1 < nkt0);
            float m = -INFINITY, l = 0.f;
            bool ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bar.pre_done, 0));
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + PF_COL_S + 32 * half, v);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            split_pack(__uint_as_float(v[8 * u + 2 * e]),
                                       __uint_as_float(v[8 * u + 2 * e + 1]), hi[e], lo[e]);
                        const uint32_t off = swz128(t, 4 * half + u);
                        st_shared16(qa + 2 * PF_CHUNK + off, hi[0], hi[1], hi[2], hi[3]);
                        st_shared16(qa + 3 * PF_CHUNK + off, lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bar.qa_ready[T]);
            }
            const int32_t *pt_row = a.page_table + (size_t)b * a.max_pages;
            int32_t page_next = pt_row[0];
            for (int kt = 0; kt < tt.nkt && ok; ++kt) {
                const int key0 = kt * PF_BN;
                const int32_t page = page_next;  // read one tile ahead, off the critical path
                if (kt + 1 < tt.nkt) page_next = pt_row[(key0 + PF_BN) / a.page_size];
                if (!(ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bar.s_full[T], kt & 1)))) break;
                tc_fence_after();
                float s[64];
                {
                    uint32_t v[32];
                    tmem_ld32(lane_base + PF_COL_S, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(v[j]);
                    tmem_ld32(lane_base + PF_COL_S + 32, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[32 + j] = __uint_as_float(v[j]);
                }
                const int klim = (page >= 0 && page < a.num_pages) ? lim - key0 : -1;
                if (klim < PF_BN - 1) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) s[j] = (j <= klim) ? s[j] : -INFINITY;
                }
                // row maximum of the raw scores (the scale is positive): eight
                // chains of three-input max, then a tree
                float m8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    m8[k] = max3f(max3f(s[k], s[8 + k], s[16 + k]), max3f(s[24 + k], s[32 + k], s[40 + k]),
                                  fmaxf(s[48 + k], s[56 + k]));
                const float mx = a.scale_log2 * max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]),
                                                      fmaxf(m8[6], m8[7]));
                const float m_new = (mx > m + kPfLazyMax) ? mx : m;
                const float alpha = (m_new == m) ? 1.f : ex2_approx(m - m_new);
                uint32_t pk[32];
                float sum = 0.f;
                if (m_new == -INFINITY) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) pk[j] = 0u;
                } else {
                    // e_j = 2^(s_j scale - m_new), two per packed FMA
                    const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2), nm2 = f2_pack(-m_new, -m_new);
                    uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(s[2 * j], s[2 * j + 1]), sc2, nm2), x0, x1);
                        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
                        pk[j] = pack_bf16(e0, e1);
                        acc[j & 3] = f2_add(acc[j & 3], f2_pack(e0, e1));
                    }
                    float u0, u1, u2, u3;
                    f2_unpack(f2_add(acc[0], acc[1]), u0, u1);
                    f2_unpack(f2_add(acc[2], acc[3]), u2, u3);
                    sum = (u0 + u1) + (u2 + u3);
                }
                l = l * alpha + sum;
                m = m_new;
                if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // the running maximum moved: rescale this row of O (the value
                    // MMA of key tile kt-1 completed before these scores did)
#pragma unroll 1
                    for (int c = 0; c < NO_LD; ++c) {
                        uint32_t v[32];
                        tmem_ld32(lane_base + 32 * c, v);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
                        tmem_st32(lane_base + 32 * c, v);
                    }
                }
                tmem_st32(lane_base + PF_COL_S, pk);  // probabilities over the scores
                if (clears && kt == nkt - 1 && max_p + 1 - key0 < PF_BN) {
                    // keys past every row of the CTA: clear their value rows
                    const int vs = kt % PF_VST;
                    if (!(ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bar.v_full[vs], (kt / PF_VST) & 1))))
                        break;
                    const int z0 = max_p + 1 - key0, units = (PF_BN - z0) * 8;
                    uint8_t *vb = smem + PF_OFF_V + vs * PF_STAGE + z0 * 128;
                    for (int u = t; u < 3 * units; u += PF_BM) {
                        const int box = u / units, w = u - box * units;
                        st_shared16(vb + box * PF_BOX + w * 16, 0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                mbar_arrive(&bar.p_full[T]);
            }
            if (ok)
                ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bar.pv_done[T], (tt.nkt - 1) & 1));
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            if (ok) {
                // (O_R / l) split into bf16 halves, K-major, over this tile's q chunks
                tc_fence_after();
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
                            const float x1 =
                                col + 1 < a.r ? __uint_as_float(v[8 * u + 2 * e + 1]) * inv_l : 0.f;
                            split_pack(x0, x1, hi[e], lo[e]);
                        }
                        const uint32_t off = swz128(t, 4 * half + u);
                        st_shared16(qa + off, hi[0], hi[1], hi[2], hi[3]);
                        st_shared16(qa + PF_CHUNK + off, lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bar.ex_ready[T]);
                ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bar.ex_done[T], 0));
            }
            if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t vo[32], ve[32];
                    tmem_ld32(lane_base + 32 * c, vo);
                    tmem_ld32(lane_base + PF_COL_E + 32 * c, ve);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float y0 = __uint_as_float(vo[2 * e]) * inv_l + __uint_as_float(ve[2 * e]);
                        const float y1 =
                            __uint_as_float(vo[2 * e + 1]) * inv_l + __uint_as_float(ve[2 * e + 1]);
                        pk[e] = row_ok ? pack_bf16(y0, y1) : 0u;
                    }
                    if (t < tt.nrows) {
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
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
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
    return launch_pdl(prefill_tc_kernel<R16>, grid, dim3(PF_THREADS), PF_SMEM, s, maps, a);
}

}  // namespace

// Shape checks and tensor maps of one call; false when the shape is not covered.
static bool prefill_tc_plan(const PrefillTcArgs &p, PfMaps &maps, int &n_pairs) {
    const lrkv_cache_t &c = p.cache;
    if (c.dtype != LRKV_BF16 || c.d_h != 128 || c.r < 8 || c.r > 64 || c.r % 8 != 0 ||
        c.page_size % PF_BN != 0 || c.H > 65535 || p.B > 65535 || p.n < 1 || p.max_ctx < 1)
        return false;
    const int64_t rows = (int64_t)c.num_pages * c.page_size;
    const int64_t max_len = (int64_t)p.max_pages * c.page_size;
    if (rows + PF_BN >= INT32_MAX || max_len >= INT32_MAX) return false;
    n_pairs = (std::min(p.n, p.max_ctx) + 2 * PF_BM - 1) / (2 * PF_BM);
    if (n_pairs > 65535) return false;
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
    int n_pairs = 0;
    if (!prefill_tc_plan(p, maps, n_pairs)) return 1;
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
    a.n_pairs = n_pairs;
    a.scale_log2 = 1.4426950408889634f / sqrtf(128.f);
    // heaviest tile pairs (most keys) first: blockIdx.z counts pairs from the end
    const dim3 grid(c.H, p.B, n_pairs);
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
