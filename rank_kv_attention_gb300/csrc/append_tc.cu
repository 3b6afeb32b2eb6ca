// LRKV cache append for many rows (prefill) on 5th-generation tensor cores.
//
// Reading note "Low-Rank Key Value Attention", section 3, Algorithm 1: new rows
// X are projected through [W_S_K | W_S_V | U_K(all heads) | U_V(all heads)] and
// each row's four blocks are stored at its token position (page table,
// same page id in all four pools).  The projection is a dense
// [n x d] . [d x (2 d_h + 2 H r)] GEMM, run here with tcgen05 by a persistent
// grid (one CTA per SM walking the output tiles) of CTA pairs (clusters of 2,
// tcgen05 cta_group::2):
//   * output tiles are 256 rows x 256 columns: two 128-column blocks of the
//     concatenated output, each block inside one of the four segments (its
//     own weight tensor map and column offset); CTA rank c owns rows
//     [128 c, 128 c + 128) of the tile and holds weight block c (for a tile
//     of one block, its rows [64 c, 64 c + 64)), so each SM receives 32 KB
//     per K step instead of 48 (the stage stream into shared memory, not the
//     tensor core, bounds a CTA that receives all of a 128 x 256 step);
//   * warp 0 (one thread) of each CTA streams its 128 x 64 K-major tile of X
//     and its weight box by TMA (128-byte swizzle) through a 6-stage ring
//     that runs on across tiles; both CTAs' copies complete on the stage
//     barrier of rank 0;
//   * warp 1 (one thread) of rank 0 issues tcgen05.mma (kind::f16, M = 256,
//     N = 256, bf16 in, fp32 accumulate) into one of two 256-column
//     accumulators in both CTAs' tensor memory, so a tile's epilogue overlaps
//     the next tile's products; stage and accumulator completions are
//     signalled in both CTAs;
//   * warps 2-5 read an accumulator back (tcgen05.ld, one row per thread),
//     round to bf16 (or 8-bit codes) and store each row's columns straight
//     into its page slot; the destination rows of a tile are looked up while
//     its products run.
// Weights are stored output-major ([columns][d]), so both operands are K-major.
#include <algorithm>

#include "append_kernels.cuh"
#include "tc_pair.cuh"

namespace lrkv {

constexpr int TC_BM = 128, TC_BN = 128, TC_BK = 64, TC_STAGES = 6;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;  // 16 KB: this CTA's 128 rows of X
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;  // 16 KB: this CTA's 128-row weight box
constexpr int TC_STAGE = TC_A_BYTES + TC_B_BYTES;
constexpr int TC_OFF_BAR = TC_STAGES * TC_STAGE;  // full[S], empty[S], acc_full[2], acc_empty[2]
constexpr int TC_OFF_TMEM = TC_OFF_BAR + 8 * (2 * TC_STAGES + 4);
constexpr int TC_SMEM = TC_OFF_TMEM + 16 + 1024;  // + alignment slack
static_assert(TC_SMEM <= 232448, "shared memory budget");
constexpr int TC_TMEM_COLS = 512;                 // two 256-column accumulators
constexpr int TC_THREADS = 192;                   // producer, MMA, 4 epilogue warps

struct TcMaps {
    CUtensorMap x;     // X [n, d]
    CUtensorMap w[4];  // W_S_K [d_h, d], W_S_V [d_h, d], U_K [H r, d], U_V [H r, d]
};

// The output's 128-column blocks: block k lies in segment seg[k] from its
// column col[k]; tile j pairs blocks 2j and 2j + 1 (the last may be alone).
constexpr int TC_MAX_BLOCKS = 32;
struct TcBlocks {
    int nblocks, ncoltiles, nrowtiles, npairs;  // npairs: (row-tile pair, column tile) items
    int seg[TC_MAX_BLOCKS];
    int col[TC_MAX_BLOCKS];
    int width[4];
};

// Item `pt` of a cluster: row tile 2 (pt / ncoltiles) + rank (possibly past
// the last row: its rows read as zeros and are not stored), column tile
// pt % ncoltiles.
__device__ __forceinline__ void tc_tile_of(const TcBlocks &t, int pt, int rank, int &m0, int &b0, int &nb) {
    const int rp = pt / t.ncoltiles, ct = pt % t.ncoltiles;
    m0 = (2 * rp + rank) * TC_BM;
    b0 = 2 * ct;
    nb = min(2, t.nblocks - b0);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS, 1)
    append_tc_kernel(const __grid_constant__ TcMaps maps, const AppendArgsT<__nv_bfloat16> a,
                     const __grid_constant__ TcBlocks tb) {
    extern __shared__ uint8_t tc_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + TC_OFF_BAR);
    uint64_t *empty = full + TC_STAGES;
    uint64_t *acc_full = empty + TC_STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + TC_OFF_TMEM);

    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nk = a.d / TC_BK;
    const int rank = (int)cluster_ctarank();
    const int pt0 = blockIdx.x >> 1, pstep = gridDim.x >> 1;  // this cluster's items

    if (tid == 0) {
        // (full and acc_empty are used in rank 0 only)
        for (int s = 0; s < TC_STAGES; ++s) {
            mbar_init(&full[s], 1);   // rank 0's producer, plus both CTAs' bytes
            mbar_init(&empty[s], 1);  // the pair's MMAs have read the stage
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&acc_full[k], 1);
            mbar_init(&acc_empty[k], 8);  // one arrival per epilogue warp of both CTAs
        }
        fence_barrier_init();
        prefetch_tensormap(&maps.x);
        for (int k = 0; k < 4; ++k) prefetch_tensormap(&maps.w[k]);
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, TC_TMEM_COLS);
    // both CTAs' barriers are initialised before either copies into the other
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    int issued = 0;  // producer: k-steps whose copies were requested

    if (warp == 0 && lane == 0) {
        // ---- producer
        const uint32_t full0 = mapa_rank(&full[0], 0);
        int it = 0;
        for (int pt = pt0; pt < tb.npairs && ok; pt += pstep) {
            int m0, b0, nb;
            tc_tile_of(tb, pt, rank, m0, b0, nb);
            // this CTA's half of B: block b0 + rank, or for a one-block tile
            // that block's rows from 64 rank (the MMA reads 64 rows per CTA)
            const int bb = nb == 2 ? b0 + rank : b0;
            const int brow = tb.col[bb] + (nb == 2 ? 0 : 64 * rank);
            const CUtensorMap *wm = &maps.w[tb.seg[bb]];
            for (int kt = 0; kt < nk; ++kt, ++it) {
                const int s = it % TC_STAGES;
                if (it >= TC_STAGES && !mbar_wait(&empty[s], ((it / TC_STAGES) - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *st = smem + s * TC_STAGE;
                const uint32_t fb = full0 + 8u * s;  // rank 0's stage barrier
                if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * TC_STAGE);
                tma_load_2d_pair(st, &maps.x, kt * TC_BK, m0, fb);
                tma_load_2d_pair(st + TC_A_BYTES, wm, kt * TC_BK, brow, fb);
                issued = it + 1;
            }
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---- MMA issuer (the pair's rows, M = 256)
        const uint32_t idesc2 = tc_idesc_bf16(2 * TC_BM, 2 * TC_BN), idesc1 = tc_idesc_bf16(2 * TC_BM, TC_BN);
        int it = 0, i = 0;
        for (int pt = pt0; pt < tb.npairs && ok; pt += pstep, ++i) {
            int m0, b0, nb;
            tc_tile_of(tb, pt, rank, m0, b0, nb);
            const int acc = i & 1;
            // the epilogue has drained this accumulator's previous tile
            if (i >= 2 && !mbar_wait(&acc_empty[acc], ((i >> 1) - 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + acc * 2 * TC_BN;
            for (int kt = 0; kt < nk; ++kt, ++it) {
                const int s = it % TC_STAGES;
                if (!mbar_wait(&full[s], (it / TC_STAGES) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + s * TC_STAGE);
                const uint64_t ad = sw128_kmajor_desc(sa), bd = sw128_kmajor_desc(sa + TC_A_BYTES);
#pragma unroll
                for (int kk = 0; kk < TC_BK / 16; ++kk)  // K = 16 per instruction: +32 bytes
                    tc2_mma_f16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2),
                                nb == 2 ? idesc2 : idesc1, (kt | kk) != 0);
                tc2_commit_both(&empty[s]);  // these products have read the stage
            }
            if (!ok) break;
            tc2_commit_both(&acc_full[acc]);  // accumulator complete
        }
    } else if (warp >= 2) {
        // ---- epilogue: thread = tile row = tensor-memory lane of its quadrant
        const int q = warp & 3, row = 32 * q + lane;
        int i = 0;
        for (int pt = pt0; pt < tb.npairs; pt += pstep, ++i) {
            int m0, b0, nb;
            tc_tile_of(tb, pt, rank, m0, b0, nb);
            // destination pool row while the products run
            int64_t dr = -1;
            {
                const int r = m0 + row;
                if (r < a.n) {
                    int32_t b, pos;
                    if (a.step_lens) {  // decode step: request r at its length - 1
                        const int32_t L = a.step_lens[r];
                        b = r;
                        pos = (L < 1 || L > a.step_max_len) ? -1 : L - 1;
                    } else {
                        b = a.seq_ids[r];
                        pos = a.positions[r];
                    }
                    if (b < 0 || b >= a.B || pos < 0 || pos >= a.max_pages * a.page_size) {
                        if (b0 == 0) status_or(a.status, LRKV_STATUS_BAD_ROW);
                    } else {
                        const int32_t page = a.page_table[(size_t)b * a.max_pages + pos / a.page_size];
                        if (page < 0 || page >= a.num_pages) {
                            if (b0 == 0) status_or(a.status, LRKV_STATUS_BAD_PAGE);
                        } else {
                            dr = (int64_t)page * a.page_size + pos % a.page_size;
                        }
                    }
                }
            }
            const int acc = i & 1;
            // tcgen05.ld is warp-collective: take the decision per warp
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], (i >> 1) & 1))) {
                if (lane == 0) status_or(a.status, LRKV_STATUS_TIMEOUT);
                break;
            }
            tc_fence_after();
            for (int k = 0; k < nb; ++k) {
                const int seg = tb.seg[b0 + k], col0 = tb.col[b0 + k], width = tb.width[seg];
                __nv_bfloat16 *base = seg == 0 ? a.S_K : seg == 1 ? a.S_V : seg == 2 ? a.R_K : a.R_V;
                const size_t rowlen = seg < 2 ? (size_t)a.d_h : (size_t)a.H * a.r;
#pragma unroll 1
                for (int c = 0; c < TC_BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + acc * 2 * TC_BN + k * TC_BN + c * 32, v);
                    const int cc = col0 + c * 32;
                    if (dr < 0 || cc >= width) continue;
                    if (a.fp8) {  // 8-bit codes of v / scale
                        uint8_t *qd = a.q8[seg] + dr * rowlen + cc;
                        const float is = a.inv_scale[seg];
                        if (cc + 32 <= width) {
                            uint32_t pk[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                pk[e] = (uint32_t)e4m3x2_from_f32(__uint_as_float(v[4 * e]) * is,
                                                                  __uint_as_float(v[4 * e + 1]) * is) |
                                        ((uint32_t)e4m3x2_from_f32(__uint_as_float(v[4 * e + 2]) * is,
                                                                   __uint_as_float(v[4 * e + 3]) * is)
                                         << 16);
                            uint4 *q4 = reinterpret_cast<uint4 *>(qd);
                            q4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            q4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        } else {
                            for (int e = 0; e < width - cc; ++e)
                                qd[e] = (uint8_t)(e4m3x2_from_f32(__uint_as_float(v[e]) * is, 0.f) & 0xffu);
                        }
                        continue;
                    }
                    __nv_bfloat16 *dst = base + dr * rowlen + cc;
                    if (cc + 32 <= width) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack_bf16(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq)
                            d4[qq] = make_uint4(pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
                    } else {
                        for (int e = 0; e < width - cc; ++e)
                            dst[e] = __float2bfloat16_rn(__uint_as_float(v[e]));
                    }
                }
            }
            // this warp has read its lanes of the accumulator
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(mapa_rank(&acc_empty[acc], 0));
        }
    }
    if (!ok) status_or(a.status, LRKV_STATUS_TIMEOUT);
    // Never leave with copies in flight into this CTA's shared memory (only
    // possible after a timeout: normally the MMA issuer consumed every stage).
    // (rank 0's stage barriers count the copies of both CTAs)
    if (warp == 0 && lane == 0 && !ok && rank == 0)
        for (int k = max(0, issued - TC_STAGES); k < issued; ++k)
            mbar_wait(&full[k % TC_STAGES], (k / TC_STAGES) & 1);
    // neither CTA leaves while the other may still copy into it or release
    // its stages
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, TC_TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// [rows, d] bf16, K (= d) innermost; box 64 x 128 with 128-byte swizzle.
// Rows beyond `rows` read as zeros.
static bool tc_map(CUtensorMap *m, const void *base, int64_t rows, int d) {
    TcEncodeFn enc = tc_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {TC_BK, 128};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The 128-column blocks of the output: per segment ceil(width / 128).
static bool tc_blocks(const AppendArgsT<__nv_bfloat16> &a, TcBlocks &t) {
    const int Hr = a.H * a.r;
    const int widths[4] = {a.d_h, a.d_h, Hr, Hr};
    t.nblocks = 0;
    for (int k = 0; k < 4; ++k) {
        t.width[k] = widths[k];
        for (int c = 0; c < widths[k]; c += TC_BN) {
            if (t.nblocks == TC_MAX_BLOCKS) return false;
            t.seg[t.nblocks] = k;
            t.col[t.nblocks] = c;
            ++t.nblocks;
        }
    }
    t.ncoltiles = (t.nblocks + 1) / 2;
    t.nrowtiles = (a.n + TC_BM - 1) / TC_BM;
    t.npairs = t.ncoltiles * ((t.nrowtiles + 1) / 2);
    return true;
}

bool tc_append_supported(int n, int d, int d_h, int H, int r) {
    // at most TC_MAX_BLOCKS 128-column blocks in the output
    const int blocks = 2 * ((d_h + TC_BN - 1) / TC_BN) + 2 * ((H * r + TC_BN - 1) / TC_BN);
    return n > 64 && d % TC_BK == 0 && d >= TC_BK && blocks <= TC_MAX_BLOCKS &&
           tc_encode() != nullptr;
}

cudaError_t launch_append_tc(const AppendArgsT<__nv_bfloat16> &a) {
    TcMaps maps;
    const int Hr = a.H * a.r;
    if (!tc_map(&maps.x, a.X, a.n, a.d) || !tc_map(&maps.w[0], a.W_S_K, a.d_h, a.d) ||
        !tc_map(&maps.w[1], a.W_S_V, a.d_h, a.d) || !tc_map(&maps.w[2], a.U_K, Hr, a.d) ||
        !tc_map(&maps.w[3], a.U_V, Hr, a.d))
        return cudaErrorInvalidValue;
    TcBlocks t;
    if (!tc_blocks(a, t)) return cudaErrorInvalidValue;
    cudaError_t e = smem_limit_once(append_tc_kernel, TC_SMEM);
    if (e != cudaSuccess) return e;
    const int grid = 2 * std::min(t.npairs, device_sm_count() / 2);
    return launch_pdl(append_tc_kernel, dim3(grid), dim3(TC_THREADS), TC_SMEM, a.stream, maps, a, t);
}

}  // namespace lrkv
