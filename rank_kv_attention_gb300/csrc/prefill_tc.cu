// Causal LRKV prefill attention on 5th-generation tensor cores.
//
// "Low-Rank Key Value Attention", section 3, equations 6-7 applied to every
// query row of a prompt chunk: for request b, head h and query row i at
// position t_i, over the request's cached rows j <= t_i,
//   s_ij = (q_i . S_K[j] + (q_i B_K[h]) . R_K[h,j]) / sqrt(d_h)
//   o_i  = sum_j a_ij S_V[j] + (sum_j a_ij R_V[h,j]) B_V[h]^T,  a_i = softmax(s_i)
// (one softmax over both score branches, section 2).  The score of a key
// tile is one accumulation
//   q . S_K^T  +  p_hi . R_K[h]^T  +  p_lo . R_K[h]^T
// where p = q B_K[h] is split into two bf16 halves (p_hi + p_lo carries ~16
// mantissa bits); the values are one contraction P . [S_V | R_V[h]] whose
// last r columns are expanded by B_V[h]^T once per query row at the end.
//
// One CTA = one (request, head, 128-row query tile); keys stream in tiles of
// 128 (two 64-row page slices; all four pools share the page id).  11 warps:
//   warps 0-7  softmax + epilogue: warps w and w+4 share the rows of tensor-
//              memory lane quadrant w%4 (thread = query row) and take key
//              columns 0..63 and 64..127 of each tile respectively;
//   warp 8     TMA producer of q, B_K, key tiles and B_V (lane 0), and owner
//              of the tensor-memory allocation;
//   warp 9     tcgen05.mma issuer (lane 0);
//   warp 10    TMA producer of value tiles (lane 0).
// Tensor memory (512 columns):
//   [0, 192)    O = [O_S | O_R] accumulator (128 + 16 ceil(r/16) columns)
//   [192, 256)  p_hi (192..223) and p_lo (224..255) as bf16 pairs: the A
//               operand of the private score branch
//   [256, 384), [384, 512)  two fp32 score buffers; the softmax overwrites the
//               first 64 columns of a buffer with the bf16 probabilities that
//               the value MMA reads as its A operand
// p = q B_K[h] is computed into the first score buffer before the loop and
// the B_V[h] expansion into it after the loop.
//
// Issue order: scores of key tile k+1, then values of tile k (after its
// softmax), so the tensor core computes the next scores while the softmax of
// the current tile runs.  tcgen05.mma runs in issue order, so the scores of
// tile k+2 (issued after the values of tile k) never overwrite probabilities
// still being read.  Softmax keeps a lazy running maximum (O is rescaled in
// tensor memory only when the maximum grows by more than 2^8).  Keys past
// every row of the CTA have their value rows cleared in shared memory, so
// whatever the cache holds there cannot reach the output.
#include <algorithm>

#include "append_kernels.cuh"
#include "tc_common.cuh"

namespace lrkv {

namespace {

constexpr int PF_BM = 128;                  // query rows per CTA
constexpr int PF_BN = 128;                  // keys per tile
constexpr int PF_HALF = 64;                 // keys per page slice / per softmax warp
constexpr int PF_BOX = PF_HALF * 128;       // one TMA box: 64 rows x 128 bytes
constexpr int PF_BLK = 2 * PF_BOX;          // 128 keys x 128 bytes
constexpr int PF_STAGE = 3 * PF_BLK;        // [S_*[:, 0:64] | S_*[:, 64:128] | R_*[h]], 48 KB
constexpr int PF_OFF_Q = 0;                 // q[:, 0:64], q[:, 64:128] (K-major)
constexpr int PF_OFF_K = 2 * PF_BM * 128;   // two key stages
constexpr int PF_OFF_V = PF_OFF_K + 2 * PF_STAGE;    // two value stages
constexpr int PF_OFF_RED = PF_OFF_V + 2 * PF_STAGE;  // bf16 row-max exchange [2][2][128]
constexpr int PF_OFF_BAR = PF_OFF_RED + 2 * 2 * PF_BM * 2;
constexpr int PF_THREADS = 352;
constexpr uint32_t PF_TMEM_COLS = 512;
constexpr uint32_t PF_COL_PQ = 192, PF_COL_S = 256;  // score buffer k at 256 + 128 k
constexpr float kPfLazyMax = 8.f;                    // log2 units

struct PfBars {
    uint64_t q_full, pre_done, qa_ready, bv_full, ex_ready, ex_done, fin;
    // a key (value) stage is free once the scores (values) of its tile are
    // complete: s_full[k] (pv_done[k]) of the tile's parity, so the
    // producers wait on those (stage k and buffer k share the index)
    uint64_t k_full[2], v_full[2];
    uint64_t s_full[2], p_full[2], pv_done[2];
    uint64_t pair[4];  // per lane quadrant: both softmax warps posted their half (64 arrivals)
    uint64_t out_ready;  // all 256 softmax threads staged their output row halves
    uint32_t tmem;
};
constexpr int PF_SMEM = PF_OFF_BAR + (int)sizeof(PfBars) + 1024;
static_assert(PF_SMEM <= 232448, "shared memory budget");

struct PfMaps {
    CUtensorMap q, out;  // Q, out [n, H, 128]: box 64 x 1 x 128
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

// 2^x on the special-function unit (PTX ex2.approx.ftz: ~2 ulp; -inf -> +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

// x -> (hi, lo) with hi = bf16(x), lo = bf16(x - hi), packed in pairs.
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - bf16lo(hi), x1 - bf16hi(hi));
}

template <int R16>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ PfMaps maps, const PfArgs a) {
    constexpr int NPV = 128 + 16 * R16;  // value columns [S_V | R_V[h] (padded)]
    extern __shared__ uint8_t pf_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(pf_smem_raw) + 1023) & ~uintptr_t(1023));
    PfBars &bar = *reinterpret_cast<PfBars *>(smem + PF_OFF_BAR);
    uint16_t *red = reinterpret_cast<uint16_t *>(smem + PF_OFF_RED);  // [slot][half][row]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, b = blockIdx.y, tq = a.n_qtiles - 1 - (int)blockIdx.z;

    if (tid == 256) {
        // (initialised by the thread that issues the first copies)
        // single arrivals (TMA transaction counts, tcgen05.commit) ...
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.pre_done, 1);
        mbar_init(&bar.bv_full, 1);
        mbar_init(&bar.ex_done, 1);
        mbar_init(&bar.fin, 1);
        for (int k = 0; k < 2; ++k) {
            mbar_init(&bar.k_full[k], 1);
            mbar_init(&bar.v_full[k], 1);
            mbar_init(&bar.s_full[k], 1);
            mbar_init(&bar.pv_done[k], 1);
            mbar_init(&bar.p_full[k], 2 * PF_BM);  // ... and arrivals of the 256 softmax threads
        }
        mbar_init(&bar.qa_ready, 2 * PF_BM);
        mbar_init(&bar.ex_ready, 2 * PF_BM);
        for (int k = 0; k < 4; ++k) mbar_init(&bar.pair[k], 64);
        mbar_init(&bar.out_ready, 2 * PF_BM);
        fence_barrier_init();
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
    const int p0 = a.start_pos[b] + (i0 - r0);                       // position of tile row 0
    const int t_lo = max(0, -p0), t_hi = min(nrows, a.max_len - p0);  // rows with a valid position
    if (t_lo >= t_hi) {  // no row of this tile has a valid position: zero its outputs
        if (tid < nrows) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((size_t)(i0 + tid) * a.H + h) * 128);
            for (int k = 0; k < 16; ++k) dst[k] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    const int max_p = p0 + t_hi - 1;  // last key position any row sees
    const int nkt = max_p / PF_BN + 1;

    if (warp == 8) {
        if (lane == 0) {
            // q tile and B_K[h] (staged in value stage 1 until p = q B_K[h] is
            // done), in flight while the tensor memory is allocated
            mbar_arrive_expect_tx(&bar.q_full, 2 * PF_BM * 128 + PF_BLK);
            tma_load_3d(smem + PF_OFF_Q, &maps.q, 0, h, i0, &bar.q_full);
            tma_load_3d(smem + PF_OFF_Q + PF_BM * 128, &maps.q, 64, h, i0, &bar.q_full);
            tma_load_2d(smem + PF_OFF_V + PF_STAGE, &maps.bk, 0, h * 128, &bar.q_full);
            tma_load_2d(smem + PF_OFF_V + PF_STAGE + PF_BOX, &maps.bk, 0, h * 128 + 64, &bar.q_full);
        }
        __syncwarp();
        tmem_alloc(&bar.tmem, PF_TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem;
    const int32_t *pt_row = a.page_table + (size_t)b * a.max_pages;

    if (warp == 8 || warp == 10) {
        if (lane == 0) {
            // ================= TMA producers: warp 8 keys, warp 10 values =================
            const bool kprod = warp == 8;
            bool ok = true;
            const int hr = h * a.r;
            // pool row of a 64-key slice of key tile kt (a fully out-of-range row,
            // which reads as zeros, for slices past the table or on an invalid page)
            auto slice_row = [&](int kt, int hh) -> int {
                const int key0 = kt * PF_BN + hh * PF_HALF;
                if (key0 / a.page_size >= a.max_pages) return -PF_HALF;
                const int32_t page = pt_row[key0 / a.page_size];
                if (page < 0 || page >= a.num_pages) {
                    if (kprod && key0 <= max_p) status_or(a.status, LRKV_STATUS_BAD_PAGE);
                    return -PF_HALF;
                }
                return page * a.page_size + key0 % a.page_size;
            };
            const CUtensorMap *m_s = kprod ? &maps.sk : &maps.sv;
            const CUtensorMap *m_r = kprod ? &maps.rk : &maps.rv;
            uint64_t *full = kprod ? bar.k_full : bar.v_full;
            uint64_t *empty = kprod ? bar.s_full : bar.pv_done;
            uint8_t *ring = smem + (kprod ? PF_OFF_K : PF_OFF_V);
            int n_iss = 0;
            int ya = slice_row(0, 0), yb = slice_row(0, 1);
            for (int kt = 0; kt < nkt; ++kt) {
                const int st = kt & 1, y0 = ya, y1 = yb;
                // page ids of the next tile: loads in flight while this one waits
                if (kt + 1 < nkt) {
                    ya = slice_row(kt + 1, 0);
                    yb = slice_row(kt + 1, 1);
                }
                // value stage 1 holds B_K[h] until p = q B_K[h] has been computed
                if ((kt >= 2 && !mbar_wait(&empty[st], ((kt >> 1) - 1) & 1)) ||
                    (!kprod && kt == 1 && !mbar_wait(&bar.pre_done, 0))) {
                    ok = false;
                    break;
                }
                uint8_t *sb = ring + st * PF_STAGE;
                mbar_arrive_expect_tx(&full[st], PF_STAGE);
                tma_load_2d(sb, m_s, 0, y0, &full[st]);
                tma_load_2d(sb + PF_BOX, m_s, 0, y1, &full[st]);
                tma_load_2d(sb + PF_BLK, m_s, 64, y0, &full[st]);
                tma_load_2d(sb + PF_BLK + PF_BOX, m_s, 64, y1, &full[st]);
                tma_load_2d(sb + 2 * PF_BLK, m_r, hr, y0, &full[st]);
                tma_load_2d(sb + 2 * PF_BLK + PF_BOX, m_r, hr, y1, &full[st]);
                ++n_iss;
            }
            // B_V[h] (K-major for the expansion) into the key stage tile nkt would use
            bool bv_issued = false;
            if (kprod && ok) {
                const int st = nkt & 1;
                if (nkt >= 2 && !mbar_wait(&bar.s_full[st], ((nkt >> 1) - 1) & 1)) {
                    ok = false;
                } else {
                    uint8_t *kb = smem + PF_OFF_K + st * PF_STAGE;
                    mbar_arrive_expect_tx(&bar.bv_full, PF_BLK);
                    tma_load_2d(kb, &maps.bv, 0, h * 128, &bar.bv_full);
                    tma_load_2d(kb + PF_BOX, &maps.bv, 0, h * 128 + 64, &bar.bv_full);
                    bv_issued = true;
                }
            }
            if (!ok) status_or(a.status, LRKV_STATUS_TIMEOUT);
            // drain: every copy issued here has landed before the CTA can exit
            if (kprod) mbar_wait(&bar.q_full, 0);
            for (int st = 0; st < 2 && st < n_iss; ++st)
                mbar_wait(&full[st], ((n_iss - 1 - st) >> 1) & 1);
            if (bv_issued) mbar_wait(&bar.bv_full, 0);
        }
    } else if (warp == 9) {
        if (lane == 0) {
            // ================= MMA issuer =================
            constexpr uint32_t id_s = tc_idesc_bf16(PF_BM, PF_BN);
            constexpr uint32_t id_pv = tc_idesc_bf16_bmn(PF_BM, NPV);
            constexpr uint32_t id_pre = tc_idesc_bf16_bmn(PF_BM, 64);
            constexpr uint32_t id_ex = tc_idesc_bf16(PF_BM, 128);
            const uint32_t base = smem_u32(smem);
            const uint32_t q0 = sw128_desc_lo(base + PF_OFF_Q, 16);
            const uint32_t q1 = sw128_desc_lo(base + PF_OFF_Q + PF_BM * 128, 16);
            const uint32_t pq = tmem + PF_COL_PQ;
            // scores of key tile kt into buffer kt & 1
            auto scores = [&](int kt) {
                const uint32_t kb = base + PF_OFF_K + (kt & 1) * PF_STAGE;
                const uint32_t k0 = sw128_desc_lo(kb, 16), k1 = sw128_desc_lo(kb + PF_BLK, 16);
                const uint32_t kr = sw128_desc_lo(kb + 2 * PF_BLK, 16);
                const uint32_t d = tmem + PF_COL_S + 128 * (kt & 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc_mma_lo(d, q0 + 2 * kk, k0 + 2 * kk, id_s, kk != 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc_mma_lo(d, q1 + 2 * kk, k1 + 2 * kk, id_s, 1);
#pragma unroll
                for (int kk = 0; kk < R16; ++kk) {  // p_hi . R_K[h] + p_lo . R_K[h]
                    tc_mma_ts_lo(d, pq + 8 * kk, kr + 2 * kk, id_s, 1);
                    tc_mma_ts_lo(d, pq + 32 + 8 * kk, kr + 2 * kk, id_s, 1);
                }
            };
            bool ok = mbar_wait(&bar.q_full, 0);
            if (ok) {
                // p = q B_K[h]: A = q (K-major), B = B_K[h] rows (MN-major, one 64-column block)
                tc_fence_after();
                const uint32_t bk = sw128_desc_lo(base + PF_OFF_V + PF_STAGE, PF_BLK);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_lo(tmem + PF_COL_S, (kk < 4 ? q0 : q1) + 2 * (kk & 3), bk + 128 * kk, id_pre,
                              kk != 0);
                tc_commit(&bar.pre_done);
                ok = mbar_wait(&bar.qa_ready, 0) && mbar_wait(&bar.k_full[0], 0);
            }
            if (ok) {
                tc_fence_after();
                scores(0);
                tc_commit(&bar.s_full[0]);
            }
            for (int kt = 0; kt < nkt && ok; ++kt) {
                const int st = kt & 1;
                if (kt + 1 < nkt) {
                    const int s1 = (kt + 1) & 1;
                    if (!mbar_wait(&bar.k_full[s1], ((kt + 1) >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    scores(kt + 1);
                    tc_commit(&bar.s_full[s1]);
                }
                if (!mbar_wait(&bar.p_full[st], (kt >> 1) & 1) ||
                    !mbar_wait(&bar.v_full[st], (kt >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t vb = sw128_desc_lo(base + PF_OFF_V + st * PF_STAGE, PF_BLK);
                const uint32_t pa = tmem + PF_COL_S + 128 * st;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // 16 keys (8 packed columns) per instruction
                    tc_mma_ts_lo(tmem, pa + 8 * kk, vb + 128 * kk, id_pv, (kt | kk) != 0);
                tc_commit(&bar.pv_done[st]);
            }
            // E = (O_R / l)_hi B_V[h]^T + (O_R / l)_lo B_V[h]^T into score buffer 0
            if (ok) ok = mbar_wait(&bar.ex_ready, 0) && mbar_wait(&bar.bv_full, 0);
            if (ok) {
                tc_fence_after();
                const uint32_t bv = sw128_desc_lo(base + PF_OFF_K + (nkt & 1) * PF_STAGE, 16);
#pragma unroll
                for (int kk = 0; kk < R16; ++kk) {
                    tc_mma_ts_lo(tmem + PF_COL_S, pq + 8 * kk, bv + 2 * kk, id_ex, kk != 0);
                    tc_mma_ts_lo(tmem + PF_COL_S, pq + 32 + 8 * kk, bv + 2 * kk, id_ex, 1);
                }
                tc_commit(&bar.ex_done);
            }
            if (!ok) status_or(a.status, LRKV_STATUS_TIMEOUT);
            tc_commit(&bar.fin);  // drain: all MMAs issued here are complete
            mbar_wait(&bar.fin, 0);
        }
    } else {
        // ================= softmax + epilogue =================
        // warp w: rows 32 (w & 3) + lane, key columns [64 hf, 64 hf + 64) of each tile
        const int q4 = warp & 3, hf = warp >> 2, t = 32 * q4 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q4) << 16);
        const bool row_ok = t >= t_lo && t < t_hi;
        const int lim = row_ok ? p0 + t : -1;  // last visible key position
        float m = -INFINITY, l = 0.f;
        // exchange with the other warp of this quadrant: phase k of bar.pair[q4]
        // completes once both warps posted their k-th value (bounded waits)
        int pair_phase = 0;
        auto pair_exchange = [&]() -> bool {
            tc_fence_before();
            mbar_arrive(&bar.pair[q4]);
            const bool got = __all_sync(0xffffffffu, mbar_wait(&bar.pair[q4], pair_phase & 1));
            ++pair_phase;
            tc_fence_after();
            return got;
        };
        bool ok = __all_sync(0xffffffffu, mbar_wait(&bar.pre_done, 0));
        if (ok) {
            // p -> bf16 halves in tensor memory: warp half 0 writes p_hi, half 1 p_lo
            tc_fence_after();
            uint32_t v[32], pk[32];
            tmem_ld32(lane_base + PF_COL_S, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                uint32_t hi, lo;
                split_pack(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]), hi, lo);
                pk[j] = hf ? lo : hi;
            }
            tmem_ld32(lane_base + PF_COL_S + 32, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                uint32_t hi, lo;
                split_pack(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]), hi, lo);
                pk[16 + j] = hf ? lo : hi;
            }
            tmem_st32(lane_base + PF_COL_PQ + 32 * hf, pk);
            tc_fence_before();
            mbar_arrive(&bar.qa_ready);
        }
        int32_t page_next = pt_row[min(hf * PF_HALF / a.page_size, a.max_pages - 1)];
        for (int kt = 0; kt < nkt && ok; ++kt) {
            const int st = kt & 1, key0 = kt * PF_BN + hf * PF_HALF;
            const int32_t page = page_next;  // read one tile ahead, off the critical path
            if (kt + 1 < nkt) page_next = pt_row[min((key0 + PF_BN) / a.page_size, a.max_pages - 1)];
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full[st], (kt >> 1) & 1)))) break;
            tc_fence_after();
            float s[64];
            {
                uint32_t v[32];
                tmem_ld32(lane_base + PF_COL_S + 128 * st + 64 * hf, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(v[j]);
                tmem_ld32(lane_base + PF_COL_S + 128 * st + 64 * hf + 32, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) s[32 + j] = __uint_as_float(v[j]);
            }
            const int klim = (page >= 0 && page < a.num_pages) ? lim - key0 : -1;
            if (klim < PF_HALF - 1) {
#pragma unroll
                for (int j = 0; j < 64; ++j) s[j] = (j <= klim) ? s[j] : -INFINITY;
            }
            // row maximum of the raw scores (the scale is positive), combined
            // with the other half of the row through shared memory
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                m8[k] = max3f(max3f(s[k], s[8 + k], s[16 + k]), max3f(s[24 + k], s[32 + k], s[40 + k]),
                              fmaxf(s[48 + k], s[56 + k]));
            // both halves use the bf16-rounded maxima, so they agree exactly on the
            // running maximum (any reference point works for the softmax)
            const __nv_bfloat16 mh = __float2bfloat16_rn(
                max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            red[(st * 2 + hf) * PF_BM + t] = __bfloat16_as_ushort(mh);
            // also orders both halves' score reads before the probability writes
            if (!(ok = pair_exchange())) break;
            const float mx = a.scale_log2 * fmaxf(__bfloat162float(mh),
                                                  __bfloat162float(__ushort_as_bfloat16(
                                                      red[(st * 2 + (hf ^ 1)) * PF_BM + t])));
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
            l = l * alpha + sum;  // this half's share of the row sum
            m = m_new;
            if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // the running maximum moved: once the values of tile kt-1 are
                // in, rescale this half's 96 columns of the O row
                if (!(ok = __all_sync(0xffffffffu,
                                      mbar_wait(&bar.pv_done[st ^ 1], ((kt - 1) >> 1) & 1))))
                    break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 3; ++c) {
                    uint32_t v[32];
                    const uint32_t col = 96 * hf + 32 * c;
                    tmem_ld32(lane_base + col, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
                    tmem_st32(lane_base + col, v);
                }
            }
            tmem_st32(lane_base + PF_COL_S + 128 * st + 32 * hf, pk);  // probabilities over the scores
            if (kt == nkt - 1 && max_p + 1 - kt * PF_BN < PF_BN) {
                // keys past every row of the CTA: clear their value rows
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.v_full[st], (kt >> 1) & 1)))) break;
                const int z0 = max_p + 1 - kt * PF_BN;  // 1..127
                uint8_t *vb = smem + PF_OFF_V + st * PF_STAGE;
                // 3 blocks x (128 - z0) rows x 8 16-byte units; key j of a block
                // sits in 64-row box j / 64, row j % 64
                const int units = (PF_BN - z0) * 8;
                for (int u = tid; u < 3 * units; u += 2 * PF_BM) {
                    const int blk = u / units, w = u - blk * units, key = z0 + (w >> 3);
                    *reinterpret_cast<uint4 *>(vb + blk * PF_BLK + (key >> 6) * PF_BOX + (key & 63) * 128 +
                                               (w & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(&bar.p_full[st]);
        }
        if (ok)
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.pv_done[(nkt - 1) & 1], ((nkt - 1) >> 1) & 1));
        // row sum of both halves, exchanged through the q tile (no longer read:
        // the last scores completed before this softmax began)
        float *lsum = reinterpret_cast<float *>(smem + PF_OFF_Q);
        lsum[hf * PF_BM + t] = l;
        if (ok) ok = pair_exchange();
        const float lt = l + lsum[(hf ^ 1) * PF_BM + t];
        const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
        if (ok) {
            // (O_R / l) in bf16 halves over p's columns: half 0 the high part, half 1 the low part
            tc_fence_after();
            uint32_t v[32], pk[32];
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                tmem_ld32(lane_base + 128 + 32 * g, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int col = 32 * g + 2 * j;
                    const float x0 = col < a.r ? __uint_as_float(v[2 * j]) * inv_l : 0.f;
                    const float x1 = col + 1 < a.r ? __uint_as_float(v[2 * j + 1]) * inv_l : 0.f;
                    uint32_t hi, lo;
                    split_pack(x0, x1, hi, lo);
                    pk[16 * g + j] = hf ? lo : hi;
                }
            }
            tmem_st32(lane_base + PF_COL_PQ + 32 * hf, pk);
            tc_fence_before();
            mbar_arrive(&bar.ex_ready);
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.ex_done, 0));
        }
        if (ok) {
            tc_fence_after();
            // a full tile is staged in the q buffer (TMA swizzle layout, half hf
            // holds output columns 64 hf .. 64 hf + 63) and written by two TMA
            // stores; a partial tile (whose box would cover the next request's
            // rows) is written row by row
            const bool full = nrows == PF_BM;
            uint8_t *stage = smem + PF_OFF_Q + hf * (PF_BM * 128);
            __nv_bfloat16 *dst = a.out + ((size_t)(i0 + t) * a.H + h) * 128 + 64 * hf;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                uint32_t vo[32], ve[32];
                tmem_ld32(lane_base + 64 * hf + 32 * c, vo);
                tmem_ld32(lane_base + PF_COL_S + 64 * hf + 32 * c, ve);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float y0 = __uint_as_float(vo[2 * e]) * inv_l + __uint_as_float(ve[2 * e]);
                    const float y1 = __uint_as_float(vo[2 * e + 1]) * inv_l + __uint_as_float(ve[2 * e + 1]);
                    pk[e] = row_ok ? pack_bf16(y0, y1) : 0u;
                }
                if (full) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4 *>(stage + swz128(t, 4 * c + k)) =
                            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                } else if (t < nrows) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        d4[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
            }
            if (full) {
                fence_proxy_async_smem();
                mbar_arrive(&bar.out_ready);
                if (tid == 0) {
                    if (mbar_wait(&bar.out_ready, 0)) {
                        tma_store_3d(&maps.out, 0, h, i0, smem + PF_OFF_Q);
                        tma_store_3d(&maps.out, 64, h, i0, smem + PF_OFF_Q + PF_BM * 128);
                        bulk_commit_group();
                        bulk_wait_read_all();
                    } else {
                        status_or(a.status, LRKV_STATUS_TIMEOUT);
                    }
                }
            }
        } else if (lane == 0) {
            status_or(a.status, LRKV_STATUS_TIMEOUT);
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
    cudaError_t e = smem_limit_once(prefill_tc_kernel<R16>, PF_SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(prefill_tc_kernel<R16>, grid, dim3(PF_THREADS), PF_SMEM, s, maps, a);
}

}  // namespace

// Shape checks and tensor maps of one call; false when the shape is not covered.
static bool prefill_tc_plan(const PrefillTcArgs &p, PfMaps &maps, int &n_qtiles) {
    const lrkv_cache_t &c = p.cache;
    if (c.dtype != LRKV_BF16 || c.N_K || cache_groups(c) != 1 || c.d_h != 128 || c.r < 8 || c.r > 64 || c.r % 8 != 0 ||
        c.page_size % PF_HALF != 0 || c.H > 65535 || p.B > 65535 || p.n < 1 || p.max_ctx < 1)
        return false;
    const int64_t rows = (int64_t)c.num_pages * c.page_size;
    const int64_t max_len = (int64_t)p.max_pages * c.page_size;
    if (rows + PF_HALF >= INT32_MAX || max_len >= INT32_MAX) return false;
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
           tma_map_bf16(&maps.out, p.out, 3, qdims, qstr, qbox) &&
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
    p.out = const_cast<void *>(cache.S_K);
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
