// LRKV cache append for many rows (prefill) on 5th-generation tensor cores.
//
// Reading note "Low-Rank Key Value Attention", section 3, Algorithm 1: new rows
// X are projected through [W_S_K | W_S_V | U_K(all heads) | U_V(all heads)] and
// each row's four blocks are stored at its token position (page table,
// same page id in all four pools).  The projection is a dense
// [n x d] . [d x (2 d_h + 2 H r)] GEMM, run here with tcgen05:
//   * one CTA per 128-row x 128-column output tile, 4 warps;
//   * warp 0 (one thread) streams 128 x 64 K-major tiles of X and of the
//     weight segment by TMA (128-byte swizzle) through a 4-stage ring;
//   * warp 1 (one thread) issues tcgen05.mma (kind::f16, bf16 in, fp32
//     accumulate) into a 128 x 128 fp32 accumulator in tensor memory and
//     releases each stage with tcgen05.commit;
//   * all 4 warps then read the accumulator back (tcgen05.ld, one row per
//     thread), round to bf16 and store each row's 128 columns straight into
//     its page slot.
// Weights are stored output-major ([columns][d]), so both operands are K-major.
#include "append_kernels.cuh"
#include "tc_common.cuh"

namespace lrkv {

constexpr int TC_BM = 128, TC_BN = 128, TC_BK = 64, TC_STAGES = 4;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;  // 16 KB
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;  // 16 KB
constexpr int TC_STAGE = TC_A_BYTES + TC_B_BYTES;
constexpr int TC_OFF_BAR = TC_STAGES * TC_STAGE;          // full[S], empty[S], accum
constexpr int TC_OFF_TMEM = TC_OFF_BAR + 8 * (2 * TC_STAGES + 1);
constexpr int TC_OFF_ROWS = TC_OFF_TMEM + 8;               // int64 destination rows [128]
constexpr int TC_SMEM = TC_OFF_ROWS + 8 * TC_BM + 1024;    // + alignment slack
constexpr int TC_TMEM_COLS = 128;

struct TcMaps {
    CUtensorMap x;     // X [n, d]
    CUtensorMap w[4];  // W_S_K [d_h, d], W_S_V [d_h, d], U_K [H r, d], U_V [H r, d]
};

struct TcTiles {
    int first[5];  // first output-column tile of each segment; first[4] = total tiles
    int width[4];  // columns of each segment
};

__global__ void __launch_bounds__(128, 1)
    append_tc_kernel(const __grid_constant__ TcMaps maps, const AppendArgsT<__nv_bfloat16> a,
                     const TcTiles tiles) {
    extern __shared__ uint8_t tc_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + TC_OFF_BAR);
    uint64_t *empty = full + TC_STAGES;
    uint64_t *accum = empty + TC_STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + TC_OFF_TMEM);
    int64_t *dst_rows = reinterpret_cast<int64_t *>(smem + TC_OFF_ROWS);

    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nt = blockIdx.x, m0 = blockIdx.y * TC_BM;
    int seg = 0;
    while (seg < 3 && nt >= tiles.first[seg + 1]) ++seg;
    const int col0 = (nt - tiles.first[seg]) * TC_BN;  // first column inside the segment
    const int nk = a.d / TC_BK;

    if (tid == 0) {
        for (int s = 0; s < TC_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum, 1);
        fence_barrier_init();
        prefetch_tensormap(&maps.x);
        prefetch_tensormap(&maps.w[seg]);
    }
    if (warp == 2) tmem_alloc(tmem_slot, TC_TMEM_COLS);
    {  // destination pool row of every tile row (or -1)
        const int i = m0 + tid;
        int64_t dr = -1;
        if (i < a.n) {
            const int32_t b = a.seq_ids[i], pos = a.positions[i];
            if (b < 0 || b >= a.B || pos < 0 || pos >= a.max_pages * a.page_size) {
                status_or(a.status, LRKV_STATUS_BAD_ROW);
            } else {
                const int32_t page = a.page_table[(size_t)b * a.max_pages + pos / a.page_size];
                if (page < 0 || page >= a.num_pages) status_or(a.status, LRKV_STATUS_BAD_PAGE);
                else dr = (int64_t)page * a.page_size + pos % a.page_size;
            }
        }
        dst_rows[tid] = dr;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0 && lane == 0) {
        // ---- producer: TMA tiles of X and of the weight segment
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % TC_STAGES;
            if (kt >= TC_STAGES && !mbar_wait(&empty[s], ((kt / TC_STAGES) - 1) & 1)) {
                ok = false;
                break;
            }
            uint8_t *st = smem + s * TC_STAGE;
            mbar_arrive_expect_tx(&full[s], TC_STAGE);
            tma_load_2d(st, &maps.x, kt * TC_BK, m0, &full[s]);
            tma_load_2d(st + TC_A_BYTES, &maps.w[seg], kt * TC_BK, col0, &full[s]);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idesc = tc_idesc_bf16(TC_BM, TC_BN);
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % TC_STAGES;
            if (!mbar_wait(&full[s], (kt / TC_STAGES) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * TC_STAGE);
            const uint64_t ad = sw128_kmajor_desc(sa), bd = sw128_kmajor_desc(sa + TC_A_BYTES);
#pragma unroll
            for (int kk = 0; kk < TC_BK / 16; ++kk)  // K = 16 per instruction: +32 bytes
                tc_mma_f16(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                           (kt | kk) != 0);
            tc_commit(&empty[s]);  // stage free once these MMAs have read it
        }
        tc_commit(accum);  // accumulator complete
    }
    if (!ok) status_or(a.status, LRKV_STATUS_TIMEOUT);

    // ---- epilogue: thread = tile row = TMEM lane
    __syncwarp();
    // tcgen05.ld is warp-collective: take the decision per warp
    const bool got = __all_sync(0xffffffffu, mbar_wait(accum, 0));
    tc_fence_after();
    if (got) {
        const int64_t dr = dst_rows[tid];
        const int width = tiles.width[seg];
        __nv_bfloat16 *base = nullptr;
        size_t rowlen = 0;
        if (seg == 0) { base = a.S_K; rowlen = a.d_h; }
        else if (seg == 1) { base = a.S_V; rowlen = a.d_h; }
        else if (seg == 2) { base = a.R_K; rowlen = (size_t)a.H * a.r; }
        else { base = a.R_V; rowlen = (size_t)a.H * a.r; }
#pragma unroll 1
        for (int c = 0; c < TC_BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, v);
            const int cc = col0 + c * 32;
            if (dr < 0 || cc >= width) continue;
            if (a.fp8) {  // 8-bit codes of v / scale
                uint8_t *q = a.q8[seg] + dr * rowlen + cc;
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
                    uint4 *q4 = reinterpret_cast<uint4 *>(q);
                    q4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    q4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                } else {
                    for (int e = 0; e < width - cc; ++e)
                        q[e] = (uint8_t)(e4m3x2_from_f32(__uint_as_float(v[e]) * is, 0.f) & 0xffu);
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
                for (int q = 0; q < 4; ++q)
                    d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            } else {
                for (int e = 0; e < width - cc; ++e) dst[e] = __float2bfloat16_rn(__uint_as_float(v[e]));
            }
        }
    } else {
        status_or(a.status, LRKV_STATUS_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) tmem_dealloc(tmem, TC_TMEM_COLS);
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

bool tc_append_supported(int n, int d, int d_h, int H, int r) {
    (void)d_h; (void)H; (void)r;
    return n > 64 && d % TC_BK == 0 && d >= TC_BK && tc_encode() != nullptr;
}

cudaError_t launch_append_tc(const AppendArgsT<__nv_bfloat16> &a) {
    TcMaps maps;
    const int Hr = a.H * a.r;
    if (!tc_map(&maps.x, a.X, a.n, a.d) || !tc_map(&maps.w[0], a.W_S_K, a.d_h, a.d) ||
        !tc_map(&maps.w[1], a.W_S_V, a.d_h, a.d) || !tc_map(&maps.w[2], a.U_K, Hr, a.d) ||
        !tc_map(&maps.w[3], a.U_V, Hr, a.d))
        return cudaErrorInvalidValue;
    TcTiles t;
    const int widths[4] = {a.d_h, a.d_h, Hr, Hr};
    t.first[0] = 0;
    for (int k = 0; k < 4; ++k) {
        t.width[k] = widths[k];
        t.first[k + 1] = t.first[k] + (widths[k] + TC_BN - 1) / TC_BN;
    }
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(append_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(t.first[4], (a.n + TC_BM - 1) / TC_BM);
    return launch_pdl(append_tc_kernel, grid, dim3(128), TC_SMEM, a.stream, maps, a, t);
}

}  // namespace lrkv
