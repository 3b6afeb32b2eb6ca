// LRKV decode split kernel for bf16 caches with d_h = 128 (sm_103a).
//
// Reading note "Low-Rank Key Value Attention": section 3, Algorithm 2 and
// equations 6-7, fused as the note describes after Algorithm 2 (running max,
// exp-sum, a shared and a private value accumulator, both rescaled by the
// same factor when the max moves); section 4 on why one shared tile must be
// reused by every head for the byte savings to show.
//
// One CTA (8 warps) streams a contiguous range of cache rows, possibly
// spanning several requests (see DecodePlan), for ALL H heads:
//   * 16-row tiles are staged by TMA (cp.async.bulk.tensor, 128-byte swizzle)
//     into a ring of shared-memory stages: the shared S_K / S_V rows (read from
//     HBM once, used by every head) and the private R_K / R_V rows of all
//     heads; completion is tracked by one mbarrier per stage;
//   * every warp owns H/8 heads end to end, so no CTA-wide barrier is needed
//     per tile.  All four contractions run on tensor cores (mma.m16n8k16, bf16
//     in, fp32 accumulate), with the tile rows or the value columns as M and
//     the warp's heads as N:
//       scores  = S_K[16 x 128] . Q^T  +  R_K[16 x (H/8) r] . blockdiag(p)^T
//       values += S_V^T . P^T           and  R_V^T . P^T  (private reduction)
//     where blockdiag(p) puts each head's private query p_h = q_h B_K[h] on
//     that head's own r columns of the tile, so the private score of head h
//     only ever meets R_K[h]; p and the softmax weights P enter as bf16
//     hi + lo halves, which keeps ~16 significant bits;
//   * the online softmax runs inside half-warps (lane = (head, row)); the
//     running maximum is only moved when the tile maximum exceeds it by more
//     than 2^8, so accumulators are rarely rescaled (the result is the same:
//     numerator and denominator share the reference);
//   * a stage is refilled by the last warp that finishes it (shared counter),
//     so the copy of tile k+STAGES starts as soon as tile k is free.
// Each (request, CTA) segment writes (m, l, accS, accR) to its partial slot;
// the combine kernel merges segments and expands accR by B_V^T once.
// Kernels of one decode are launched with programmatic dependent launch:
// each waits (griddepcontrol.wait) for its predecessor before reading its
// results, so only launch latency overlaps.
#include <algorithm>

#include "decode_kernels.cuh"
#include "tc_common.cuh"

namespace lrkv {

constexpr int kLocalReq = 64;  // requests whose offsets fit in pl[16 .. 16 + kLocalReq]

// Q8_: the cache holds 8-bit E4M3 codes (one byte per element) instead of bf16.
// GS_: the scores are given (written by the rotary score kernel): a stage
// holds S_V, R_V and the tile's 16 x H fp32 scores, no S_K or R_K.
// NGRP_: shared key/value groups (a token's shared rows hold NGRP x d_h).
template <int H_, int R_, int STAGES_, bool Q8_ = false, bool GS_ = false, int NGRP_ = 1>
struct FastCfg {
    // rows per stage: given scores and 8-bit codes carry half the bytes per
    // row, so a stage holds 32 rows (two 16-row halves) to keep the cost of
    // a stage's wait and release per byte
    static constexpr int H = H_, R = R_, TS = (GS_ || Q8_) ? 32 : 16, STAGES = STAGES_;
    static constexpr bool Q8 = Q8_, GS = GS_;
    static constexpr int NGRP = NGRP_;
    static constexpr int EB = Q8 ? 1 : 2;    // bytes per cache element
    static constexpr int DH = 128;
    static constexpr int NCW = 8, NT = NCW * 32;
    static constexpr int HPW = H / NCW;      // heads per warp (2 or 4)
    static constexpr int NH = HPW / 2;       // head slots per thread
    static constexpr int RC = R / 8;         // 16-byte chunks per private row
    static constexpr int BOX = TS * 128;     // one 16-row x 128-byte swizzled box
    static constexpr int NBOX_S = NGRP * DH * EB / 128;  // all groups' shared columns
    static constexpr int GCH = DH * EB / 16;                // 16-byte chunks of one group's row
    static constexpr int NBOX_R = H * R * EB / 128;
    static constexpr int S_BYTES = NBOX_S * BOX, R_BYTES = NBOX_R * BOX;
    static constexpr int OFF_SK = 0, OFF_SV = GS ? 0 : S_BYTES, OFF_RK = 2 * S_BYTES;
    static constexpr int OFF_RV = GS ? S_BYTES : 2 * S_BYTES + R_BYTES;
    // joint key norms (optional): the tile's 16 x H bf16 reciprocals
    static constexpr int OFF_NK = 2 * S_BYTES + 2 * R_BYTES;
    static constexpr int NK_TX = TS * H * 2;   // bytes one copy lands
    // given scores: the tile's 16 x H fp32 scores after S_V and R_V
    static constexpr int OFF_SC = S_BYTES + R_BYTES;
    static constexpr int SC_TX = TS * H * 4;
    static constexpr int STAGE_TX = GS ? S_BYTES + R_BYTES : 2 * S_BYTES + 2 * R_BYTES;
    static constexpr int STAGE = STAGE_TX + (GS ? (SC_TX + 1023) / 1024 * 1024 : (NK_TX + 1023) / 1024 * 1024);
    static constexpr int KSP = HPW * R / 16;  // k-steps (and m-tiles) of a warp's private columns
    static constexpr int OFF_BAR = STAGES * STAGE;   // full[STAGES]
    static constexpr int OFF_CNT = OFF_BAR + 64;     // release counters[STAGES]
    static constexpr int OFF_OK = OFF_CNT + 64;      // per-stage "page id valid" flags
    static constexpr int OFF_CUR = OFF_OK + 64;      // issue cursor
    static constexpr int OFF_PLAN = OFF_CUR + 64;    // local plan: scan scratch + request offsets
    static constexpr int OFF_PEND = OFF_PLAN + 512;  // given scores: rows of the first copies
    static constexpr int SMEM = OFF_PEND + 64 + 1024;  // + alignment slack
    // registers per thread: at most 224 leaves room for a 128-thread prologue
    // block of up to 48 registers on the same SM, so the split CTAs do not
    // wait for the prologue to leave; the widest private rows and the 8-bit
    // tiles (whose code conversions want the registers) take all 255
    static constexpr int MAXREG = (H * R >= 1024 || Q8) ? 255 : 224;

    static_assert(H == 16 || H == 32, "two or four heads per warp");
    static_assert(R % 8 == 0 && (H * R * EB) % 128 == 0, "private rows tile into 128-byte boxes");
    static_assert(STAGES <= 8, "barrier, counter and flag arrays hold 8 stages");
    static_assert((H * 2) % 16 == 0, "16-byte TMA rows of norms");
    static_assert((HPW * R) % 16 == 0, "a warp's private columns form whole mma k-steps");
    static_assert(STAGE % 1024 == 0, "128B-swizzle boxes need 1 KB alignment");
    static_assert(!(GS && Q8), "given scores come with bf16 caches");
    static_assert(NGRP == 1 || (!Q8 && !GS && H % NGRP == 0 && (H / NGRP) % HPW == 0),
                  "a warp's heads share one group (bf16 caches)");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct FastParams {
    const __nv_bfloat16 *q;
    const int32_t *seq_lens;
    const int32_t *page_table;
    const int32_t *req_row;
    int max_pages, num_pages, page_size, B;
    float scale_log2;
    DecodeWs ws;
    int32_t *status;
    float4 sc;  // 8-bit cache: pool scales of S_K, S_V, R_K, R_V
    int norm;   // the cache holds joint key norms (a fifth copy per tile)
    int max_len;  // longest valid sequence length (longer requests are not attended)
    // rotary score kernel: operands from the prologue, scores out
    const uint16_t *wt;
    const uint16_t *qb;
    const float *wsc;
    float *sc_out;
    int step_rows;  // a decode step: the append of the new rows may run beside this kernel's start
    // the merge phase: expansion bases and the output
    const __nv_bfloat16 *B_K;
    const __nv_bfloat16 *B_V;
    __nv_bfloat16 *out;
};

struct FastMaps {
    CUtensorMap sk, sv, rk, rv;
    CUtensorMap nk;  // joint key norms, or (given scores) the score array
};

// Copy-issue cursor over the CTA's tile sequence (segments in order, 16-row
// tiles inside a segment).  Lives in shared memory; only the warp that
// releases a stage last touches it, and releases happen in tile order.
struct IssueCursor {
    int b;
    int32_t start;
    int t, t_b;
    int done, issued;
    int page_key, page_id;  // page of the last issued tile: (request, page index) -> id
};


__device__ __forceinline__ const int32_t *page_row(const FastParams &P, int b) {
    return P.page_table + (size_t)(P.req_row ? P.req_row[b] : b) * P.max_pages;
}

template <class C>
__device__ __forceinline__ void cursor_begin_segment(IssueCursor *cur, const int32_t *off,
                                                     int32_t end) {
    int b = cur->b;
    while (off[b + 1] <= cur->start) ++b;
    const int32_t base = off[b];
    cur->b = b;
    cur->t = (cur->start - base) / C::TS * C::TS;
    cur->t_b = min(end, off[b + 1]) - base;
}

// Pool row of the cursor's next tile (page looked up once per page), with the
// stage's "page id valid" flag set for the consumers.
__device__ __forceinline__ int cursor_row(IssueCursor *cur, const FastParams &P, int *okf, int s) {
    // one page-table read per page (a page holds several 16-row tiles)
    const int pidx = cur->t / P.page_size;
    const int key = cur->b * P.max_pages + pidx;
    int32_t page;
    if (key == cur->page_key) {
        page = cur->page_id;
    } else {
        const int32_t *row_pt = page_row(P, cur->b);
        page = row_pt[pidx];
        cur->page_key = key;
        cur->page_id = page;
        if (pidx + 1 < P.max_pages)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(row_pt + pidx + 1));
    }
    const bool ok = page >= 0 && page < P.num_pages;
    if (!ok) {
        status_or(P.status, LRKV_STATUS_BAD_PAGE);
        page = 0;  // consumers mask the tile
    }
    okf[s] = ok;  // published to the consumers by the mbarrier phase
    return page * P.page_size + cur->t % P.page_size;
}

// Move the cursor past the tile just issued.
template <class C>
__device__ __forceinline__ void cursor_advance(IssueCursor *cur, const int32_t *off, int32_t end) {
    cur->issued += 1;
    cur->t += C::TS;
    if (cur->t >= cur->t_b) {
        cur->start = off[cur->b] + cur->t_b;
        if (cur->start >= end) cur->done = 1;
        else cursor_begin_segment<C>(cur, off, end);
    }
}

// Given scores: the copy of a tile's 16 x H scores (plan row srow onward).
template <class C>
__device__ __forceinline__ void issue_scores(uint8_t *st, const FastMaps &M, int32_t srow,
                                             uint64_t *bar) {
    mbar_arrive_expect_tx(bar, C::SC_TX);
    tma_load_3d(st + C::OFF_SC, &M.nk, 0, srow, 0, bar);
}

// Issue the copies of the cursor's next tile into its stage.
// `refill`: the stage was read by generic loads before (every issue except
// the first STAGES of a launch, whose stages are fresh), so those reads are
// ordered before the copy's writes.
// `pend` (given scores only): the scores do not exist yet; their plan row is
// kept in pend[stage] and the copy issued after the dependency wait.
// `pre_wait` (decode step): the append of the step's new rows may still be
// running, so a tile that holds a request's new row (its last row) is not
// copied yet; the call returns false and the caller issues it after the wait.
template <class C>
__device__ bool issue_next(IssueCursor *cur, const FastParams &P, const FastMaps &M,
                           const int32_t *off, uint8_t *smem, uint64_t *full, int *okf,
                           int32_t end, bool refill = true, int32_t *pend = nullptr,
                           bool pre_wait = false) {
    if (cur->done) return true;
    if (pre_wait && P.step_rows && cur->t + C::TS >= off[cur->b + 1] - off[cur->b]) return false;
    const int s = cur->issued % C::STAGES;
    const int row = cursor_row(cur, P, okf, s);
    uint8_t *st = smem + s * C::STAGE;
    if (refill) fence_proxy_async_smem();
    // each map is 3-D (64 columns, rows, 64-column block) with a box of
    // 64 x 16 x all blocks, so one copy lands the whole 16-row tile as
    // consecutive 16-row x 128-byte swizzled boxes
    // the cache streams through once per step: evict it from L2 first
    const uint64_t pol = l2_evict_first_policy();
    if constexpr (C::GS) {
        mbar_arrive_expect_tx(&full[s], C::STAGE_TX);
        tma_load_3d_hint(st + C::OFF_SV, &M.sv, 0, row, 0, &full[s], pol);
        tma_load_3d_hint(st + C::OFF_RV, &M.rv, 0, row, 0, &full[s], pol);
        const int32_t srow = off[cur->b] + cur->t;
        if (pend) pend[s] = srow;
        else issue_scores<C>(st, M, srow, &full[s]);
    } else {
        mbar_arrive_expect_tx(&full[s], C::STAGE_TX + (P.norm ? C::NK_TX : 0));
        tma_load_3d_hint(st + C::OFF_SK, &M.sk, 0, row, 0, &full[s], pol);
        tma_load_3d_hint(st + C::OFF_SV, &M.sv, 0, row, 0, &full[s], pol);
        tma_load_3d_hint(st + C::OFF_RK, &M.rk, 0, row, 0, &full[s], pol);
        tma_load_3d_hint(st + C::OFF_RV, &M.rv, 0, row, 0, &full[s], pol);
        if (P.norm) tma_load_3d_hint(st + C::OFF_NK, &M.nk, 0, row, 0, &full[s], pol);
    }
    cursor_advance<C>(cur, off, end);
    return true;
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16 *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}

// The running maximum (log2 units) only moves when a tile exceeds it by this
// much; weights stay below 2^kLazyMax, far inside fp32 range.
constexpr float kLazyMax = 8.f;

// Byte offset, inside a stage region made of 64-column swizzled boxes, of the
// 16-byte chunk `cc` (counted along the row) of tile row `j`.
__device__ __forceinline__ uint32_t box_chunk(int j, int cc) {
    return (uint32_t)((cc >> 3) * (16 * 128)) + swz128(j, cc & 7);
}

// Byte offset, inside a region of 64-column swizzled boxes of TS rows, of the
// 16-byte chunk `cc` (counted along the row) of row `j`.
template <int TS>
__device__ __forceinline__ uint32_t box_chunk_rows(int j, int cc) {
    return (uint32_t)((cc >> 3) * (TS * 128)) + swz128(j, cc & 7);
}

// ---------------------------------------------------------------------------
// 8-bit (E4M3) cache tiles.  A 16-row tile arrives as 128-byte swizzled boxes
// of codes (one box for S_K or S_V, H r / 128 for R_K or R_V).  The codes are
// widened to f16 in registers (exact: every E4M3 value is an f16 value) and
// enter f16 mma.sync with fp32 accumulation; the pool scales multiply the
// fp32 results.
//   * Scores: the order of the 16 contraction indices of a k-step is free as
//     long as both operands use the same one, so thread tq takes bytes
//     4tq .. 4tq+3 of each 16-byte chunk (one 32-bit shared load per row) for
//     its fragment slots 2tq, 2tq+1, 2tq+8, 2tq+9.
//   * Values: the tile rows stay in order (they meet the softmax weights);
//     the value columns are permuted instead: a 32-bit load at byte
//     32u + 4gq of a row holds, in order, columns gq and gq + 8 of m-tile 2u
//     and columns gq and gq + 8 of m-tile 2u + 1, and byte permutes pair the
//     rows 2tq, 2tq + 1 (and 2tq + 8, 2tq + 9) of each column into one f16x2
//     fragment register.  A trailing odd m-tile uses 16-bit loads.  Row masks
//     (invalid rows may hold any code) are applied on partial tiles only.
//   * q and p enter as f16 after an exact power-of-two scaling per head that
//     brings the head's largest |value| into [2^14, 2^15); the softmax weights
//     (at most 2^8 under the lazy maximum) enter as f16 directly.
// ---------------------------------------------------------------------------

template <class C>
__device__ __forceinline__ void q8_segment_setup(const FastParams &P, int b, int warp, int gq,
                                                 int tq, uint32_t (&qb)[8][2],
                                                 uint32_t (&pb)[C::KSP][2], float (&fS)[2],
                                                 float (&fR)[2], const float *pw) {
    // column n = gq of the B fragments is head warp*HPW + n (n < HPW), else 0;
    // contraction index k of k-step ks in slot order is 16 ks + 4 tq + e
    const bool own = gq < C::HPW;
    const __nv_bfloat16 *qrow = P.q + ((size_t)b * C::H + warp * C::HPW + (own ? gq : 0)) * C::DH;
    float qv[8][4], pv[C::KSP][4];
    float mq = 0.f, mp = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint2 u = own ? *reinterpret_cast<const uint2 *>(qrow + ks * 16 + 4 * tq) : make_uint2(0u, 0u);
        qv[ks][0] = __uint_as_float(u.x << 16);
        qv[ks][1] = __uint_as_float(u.x & 0xffff0000u);
        qv[ks][2] = __uint_as_float(u.y << 16);
        qv[ks][3] = __uint_as_float(u.y & 0xffff0000u);
#pragma unroll
        for (int e = 0; e < 4; ++e) mq = fmaxf(mq, fabsf(qv[ks][e]));
    }
    // blockdiag(p)^T: entry (k, n) is p[head n][k - n R] when k lies in head
    // n's columns of the warp, else 0 (pw: the warp's heads' p, R apart)
#pragma unroll
    for (int ks = 0; ks < C::KSP; ++ks)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = ks * 16 + 4 * tq + e;
            pv[ks][e] = (own && k / C::R == gq) ? pw[k] : 0.f;
            mp = fmaxf(mp, fabsf(pv[ks][e]));
        }
    // the head's maxima over its four lanes (same gq)
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
        mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, o));
    }
    const int eq = f16_range_shift(mq), ep = f16_range_shift(mp);
    const float uq = exp2i(eq), up = exp2i(ep);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        qb[ks][0] = pack_f16(qv[ks][0] * uq, qv[ks][1] * uq);
        qb[ks][1] = pack_f16(qv[ks][2] * uq, qv[ks][3] * uq);
    }
#pragma unroll
    for (int ks = 0; ks < C::KSP; ++ks) {
        pb[ks][0] = pack_f16(pv[ks][0] * up, pv[ks][1] * up);
        pb[ks][1] = pack_f16(pv[ks][2] * up, pv[ks][3] * up);
    }
    // factors of accumulator columns 2tq and 2tq + 1 (held by lanes 8tq, 8tq + 4)
    const float fq = P.sc.x * exp2i(-eq), fp = P.sc.z * exp2i(-ep);
    fS[0] = __shfl_sync(0xffffffffu, fq, 8 * tq);
    fS[1] = __shfl_sync(0xffffffffu, fq, 8 * tq + 4);
    fR[0] = __shfl_sync(0xffffffffu, fp, 8 * tq);
    fR[1] = __shfl_sync(0xffffffffu, fp, 8 * tq + 4);
}

__device__ __forceinline__ uint32_t lds_u32(const uint8_t *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}
__device__ __forceinline__ uint32_t lds_u16(const uint8_t *p) {
    return *reinterpret_cast<const uint16_t *>(p);
}
__device__ __forceinline__ uint32_t f16x2_lo(uint32_t w) { return f16x2_from_e4m3x2((uint16_t)w); }
__device__ __forceinline__ uint32_t f16x2_hi(uint32_t w) {
    return f16x2_from_e4m3x2((uint16_t)(w >> 16));
}

// Scores of a tile: c[row x head] = fS . (S_K . Q^T) + fR . (R_K . blockdiag(p)^T).
// rb: first stage row of the 16-row half being scored.
template <class C>
__device__ __forceinline__ void q8_scores(const uint8_t *st, int rb, int warp, int gq, int tq,
                                          const uint32_t (&qb)[8][2],
                                          const uint32_t (&pb)[C::KSP][2], const float (&fS)[2],
                                          const float (&fR)[2], float (&c)[4]) {
    float c1[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f}, c3[4] = {0.f, 0.f, 0.f, 0.f};
    const uint8_t *sk = st + C::OFF_SK, *rk = st + C::OFF_RK;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t w0 = lds_u32(sk + box_chunk_rows<C::TS>(rb + gq, ks) + 4 * tq);
        const uint32_t w1 = lds_u32(sk + box_chunk_rows<C::TS>(rb + gq + 8, ks) + 4 * tq);
        const uint32_t a[4] = {f16x2_lo(w0), f16x2_lo(w1), f16x2_hi(w0), f16x2_hi(w1)};
        if (ks & 1) mma_f16_16816(c1, a, qb[ks][0], qb[ks][1]);
        else mma_f16_16816(c, a, qb[ks][0], qb[ks][1]);
    }
    const int cw = warp * (C::HPW * C::R / 16);  // first 16-byte chunk of the warp's columns
#pragma unroll
    for (int ks = 0; ks < C::KSP; ++ks) {
        const uint32_t w0 = lds_u32(rk + box_chunk_rows<C::TS>(rb + gq, cw + ks) + 4 * tq);
        const uint32_t w1 = lds_u32(rk + box_chunk_rows<C::TS>(rb + gq + 8, cw + ks) + 4 * tq);
        const uint32_t a[4] = {f16x2_lo(w0), f16x2_lo(w1), f16x2_hi(w0), f16x2_hi(w1)};
        if (ks & 1) mma_f16_16816(c3, a, pb[ks][0], pb[ks][1]);
        else mma_f16_16816(c2, a, pb[ks][0], pb[ks][1]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) c[e] = fS[e & 1] * (c[e] + c1[e]) + fR[e & 1] * (c2[e] + c3[e]);
}

// A fragments of two value m-tiles from the 32-bit words of rows 2tq, 2tq+1,
// 2tq+8, 2tq+9 (see the layout note above); MASK: zero invalid rows.
template <bool MASK>
__device__ __forceinline__ void q8_pair_frags(uint32_t w0, uint32_t w1, uint32_t w8, uint32_t w9,
                                              uint32_t m01, uint32_t m89, uint32_t (&a)[4],
                                              uint32_t (&b)[4]) {
    const uint32_t x01 = prmt<0x5140>(w0, w1), y01 = prmt<0x7362>(w0, w1);
    const uint32_t x89 = prmt<0x5140>(w8, w9), y89 = prmt<0x7362>(w8, w9);
    a[0] = f16x2_lo(x01); a[1] = f16x2_hi(x01); a[2] = f16x2_lo(x89); a[3] = f16x2_hi(x89);
    b[0] = f16x2_lo(y01); b[1] = f16x2_hi(y01); b[2] = f16x2_lo(y89); b[3] = f16x2_hi(y89);
    if (MASK) {
        a[0] &= m01; a[1] &= m01; a[2] &= m89; a[3] &= m89;
        b[0] &= m01; b[1] &= m01; b[2] &= m89; b[3] &= m89;
    }
}

// Values of a tile: accS += S_V^T . P^T, accR += R_V^T(warp columns) . P^T.
// rb: first stage row of the 16-row half being reduced.
template <class C, bool MASK>
__device__ __forceinline__ void q8_values(const uint8_t *st, int rb, int warp, int gq, int tq,
                                          uint32_t m01, uint32_t m89, uint32_t b0, uint32_t b1,
                                          float (&accS)[8][4], float (&accR)[C::KSP][4]) {
    const uint8_t *sv = st + C::OFF_SV, *rv = st + C::OFF_RV;
    const int r0 = rb + 2 * tq, r1 = r0 + 1, r8 = r0 + 8, r9 = r0 + 9;
    auto bc = [](int j, int ch) { return box_chunk_rows<C::TS>(j, ch); };
    auto pair = [&](const uint8_t *t, int cb, float (&d0)[4], float (&d1)[4]) {
        const int ch = cb >> 4, o = cb & 15;
        uint32_t a[4], a2[4];
        q8_pair_frags<MASK>(lds_u32(t + bc(r0, ch) + o), lds_u32(t + bc(r1, ch) + o),
                            lds_u32(t + bc(r8, ch) + o), lds_u32(t + bc(r9, ch) + o),
                            m01, m89, a, a2);
        mma_f16_16816(d0, a, b0, b1);
        mma_f16_16816(d1, a2, b0, b1);
    };
#pragma unroll
    for (int u = 0; u < 4; ++u) pair(sv, 32 * u + 4 * gq, accS[2 * u], accS[2 * u + 1]);
    const int cwb = warp * C::HPW * C::R;  // first byte column of the warp's private columns
#pragma unroll
    for (int u = 0; u < C::KSP / 2; ++u) pair(rv, cwb + 32 * u + 4 * gq, accR[2 * u], accR[2 * u + 1]);
    if constexpr (C::KSP & 1) {
        constexpr int mt = C::KSP - 1;
        const int cb = cwb + 16 * mt + 2 * gq, ch = cb >> 4, o = cb & 15;
        const uint32_t h0 = lds_u16(rv + bc(r0, ch) + o), h1 = lds_u16(rv + bc(r1, ch) + o);
        const uint32_t h8 = lds_u16(rv + bc(r8, ch) + o), h9 = lds_u16(rv + bc(r9, ch) + o);
        const uint32_t x01 = prmt<0x5140>(h0, h1), x89 = prmt<0x5140>(h8, h9);
        uint32_t a[4] = {f16x2_lo(x01), f16x2_hi(x01), f16x2_lo(x89), f16x2_hi(x89)};
        if (MASK) { a[0] &= m01; a[1] &= m01; a[2] &= m89; a[3] &= m89; }
        mma_f16_16816(accR[mt], a, b0, b1);
    }
}

// Value column (relative to the tile's or the warp's first column) of
// accumulator m-tile mt, element e, under the permutation of q8_values.
template <int KSP>
__device__ __forceinline__ int q8_value_col(int mt, int e, int gq) {
    return (mt < (KSP & ~1)) ? 32 * (mt >> 1) + 4 * gq + 2 * (mt & 1) + (e >> 1)
                             : 16 * mt + 2 * gq + (e >> 1);
}

template <class C>
__device__ __forceinline__ void q8_write_partial(const FastParams &P, size_t slot, int warp, int gq,
                                                 int tq, const float (&accS)[8][4],
                                                 const float (&accR)[C::KSP][4]) {
    const size_t W = C::DH + C::R;
    float *acc = P.ws.acc;
    if (2 * tq < C::HPW) {
        const int h0 = warp * C::HPW + 2 * tq;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                acc[(slot * C::H + h0 + (e & 1)) * W + q8_value_col<8>(mt, e, gq)] = accS[mt][e] * P.sc.y;
    }
#pragma unroll
    for (int mt = 0; mt < C::KSP; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int pc = q8_value_col<C::KSP>(mt, e, gq);
            const int n = 2 * tq + (e & 1);
            if (n < C::HPW && pc / C::R == n)
                acc[(slot * C::H + warp * C::HPW + n) * W + C::DH + (pc - n * C::R)] = accR[mt][e] * P.sc.w;
        }
}

// ---------------------------------------------------------------------------
// Local launch plan of CTA g out of G: the rows of all requests laid end to
// end, cut into G chunks of whole 16-row tiles, with the same validated
// lengths and chunk formula as the prologue's plan.  It reads only caller
// inputs (sequence lengths, page table), which were complete before the
// prologue kernel got past its own wait and let the next grid launch, so the
// first tiles can be requested while the prologue is still computing.  Every
// thread calls it; a CTA without rows gets start >= end (before any barrier
// that a CTA with rows would pass).  When the CTA's requests do not fit the
// local offset table, it waits for the prologue and uses its offsets.
// pl (shared, >= 96 ints): [0] first request [1] last request [2] first page
// key [3] first page id [4 .. 4 + warps) scan sums [16 ..] request offsets.
// ---------------------------------------------------------------------------
struct CtaRange {
    int b0;
    int32_t start, end;
    const int32_t *off;  // off[b] for the CTA's requests
    bool local;
    int32_t chunk;       // rows per CTA: CTA g covers [g chunk, (g + 1) chunk)
};


template <int NT>
__device__ __forceinline__ CtaRange cta_range(const FastParams &P, int g, int G, int32_t *pl) {
    static_assert(NT / 32 <= 12, "scan sums fit pl[4 .. 15]");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Bn = P.B;
    const int per = (Bn + NT - 1) / NT;
    const int lo = min(Bn, tid * per), hi = min(Bn, lo + per);
    auto len_of = [&](int bb) { return streamed_len(P.seq_lens[bb], P.max_len); };
    // with at most one request per thread its length stays in a register
    const int32_t my_len = lo < hi ? len_of(lo) : 0;
    auto len_at = [&](int bb) { return (per == 1) ? my_len : len_of(bb); };
    int32_t mysum = 0;
    for (int bb = lo; bb < hi; ++bb) mysum += len_at(bb);
    int32_t incl = mysum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) pl[4 + warp] = incl;
    __syncthreads();
    int32_t wbase = 0, total = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const int32_t v = pl[4 + w];
        if (w < warp) wbase += v;
        total += v;
    }
    const int32_t base_t = wbase + incl - mysum;  // offset of request lo
    int32_t chunk = (total + G - 1) / G;
    chunk = max(chunk, kPlanTileAlign);
    chunk = (chunk + kPlanTileAlign - 1) / kPlanTileAlign * kPlanTileAlign;
    CtaRange rg;
    rg.chunk = chunk;
    rg.start = g * chunk;
    rg.end = min(total, rg.start + chunk);
    rg.b0 = 0;
    rg.off = nullptr;
    rg.local = true;
    // a batch of at most kLocalReq requests: every CTA (with rows or not)
    // keeps the whole offset table, off[b] at pl[16 + b]
    const bool all_local = Bn <= kLocalReq;
    if (all_local) {
        int32_t o = base_t;
        for (int bb = lo; bb < hi; ++bb) {
            pl[16 + bb] = o;
            o += len_at(bb);
        }
        if (hi == Bn) pl[16 + Bn] = o;  // off[B] = total
    }
    if (rg.start >= rg.end) {  // the whole CTA takes this path
        if (all_local) {
            __syncthreads();
            rg.off = pl + 16;
        }
        return rg;
    }
    {
        int32_t o = base_t;
        for (int bb = lo; bb < hi; ++bb) {
            const int32_t L = len_at(bb);
            if (L > 0 && o <= rg.start && rg.start < o + L) {
                pl[0] = bb;
                // the page of the CTA's first tile, so the copy issuer need
                // not read it after the barrier
                const int pidx = (rg.start - o) / P.page_size;
                pl[2] = bb * P.max_pages + pidx;
                pl[3] = page_row(P, bb)[pidx];
            }
            if (L > 0 && o < rg.end && rg.end <= o + L) pl[1] = bb;
            o += L;
        }
    }
    __syncthreads();
    rg.b0 = pl[0];
    if (all_local) {
        rg.off = pl + 16;
        return rg;
    }
    rg.local = pl[1] + 1 - rg.b0 <= kLocalReq;
    if (rg.local) {
        int32_t o = base_t;
        for (int bb = lo; bb < hi; ++bb) {
            if (bb >= rg.b0 && bb - rg.b0 <= kLocalReq) pl[16 + bb - rg.b0] = o;
            o += len_at(bb);
        }
        if (hi == Bn && Bn - rg.b0 <= kLocalReq) pl[16 + Bn - rg.b0] = o;  // off[B] = total
    }
    __syncthreads();
    rg.off = rg.local ? pl + 16 - rg.b0 : P.ws.off;
    if (!rg.local) pdl_wait();  // fall back to the prologue's offsets
    return rg;
}

__device__ __forceinline__ uint32_t u4w(const uint4 &v, int w) {
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Bounded wait until the workspace counter reaches the grid size (every CTA
// has written its partial states).  After ~2 s it flags LRKV_STATUS_TIMEOUT
// and returns false; the caller goes on without the data it waited for
// (wrong values, flagged, but nothing out of bounds).
__device__ __forceinline__ bool wait_grid_count(const FastParams &P) {
    const int32_t *c = P.ws.cnt;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
        if (v >= (int32_t)gridDim.x) return true;
        if (it == 0) t0 = globaltimer_ns();
        else if ((it & 63u) == 63u && globaltimer_ns() - t0 > 2000000000ull) {
            status_or(P.status, LRKV_STATUS_TIMEOUT);
            return false;
        }
        __nanosleep(128);
    }
}

template <class C>
__device__ __forceinline__ void stream_range(const FastMaps &M, const FastParams &P, const CtaRange &rg,
                                             uint8_t *smem);
template <class C>
__device__ void merge_phase(const FastParams &P, const CtaRange &rg, const int32_t *off, int warp,
                            int lane, float *scratch);

template <class C>
__global__ void __maxnreg__(C::MAXREG)
    decode_split_fast_kernel(const __grid_constant__ FastMaps M, const FastParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    int *cnt = reinterpret_cast<int *>(smem + C::OFF_CNT);
    int *okf = reinterpret_cast<int *>(smem + C::OFF_OK);
    IssueCursor *cur = reinterpret_cast<IssueCursor *>(smem + C::OFF_CUR);
    int32_t *pend = reinterpret_cast<int32_t *>(smem + C::OFF_PEND);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x;
    const DecodeWs &ws = P.ws;

    // fetch the tensor-map descriptors now: the first copies use them right
    // after the plan below
    if (tid == 32) {
        if (!C::GS) prefetch_tensormap(&M.sk);
        prefetch_tensormap(&M.sv);
        if (!C::GS) prefetch_tensormap(&M.rk);
        prefetch_tensormap(&M.rv);
        if (C::GS || P.norm) prefetch_tensormap(&M.nk);
    }
    // warm L2 with the page-table rows: the copy issuer reads them right
    // after the plan below (caller inputs, complete before this grid launched)
    if (!P.req_row) {
        const size_t pt_bytes = (size_t)P.B * P.max_pages * sizeof(int32_t);
        if (pt_bytes <= 64 * 1024)
            for (size_t o = (size_t)tid * 128; o < pt_bytes; o += (size_t)C::NT * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(P.page_table) + o));
    }
    int32_t *pl = reinterpret_cast<int32_t *>(smem + C::OFF_PLAN);
    const CtaRange rg = cta_range<C::NT>(P, g, (int)gridDim.x, pl);
    const int32_t start0 = rg.start, end = rg.end;
    const bool has_rows = start0 < end;
    const int b0 = rg.b0;
    const bool local = rg.local;
    const int32_t *off = rg.off;  // off[b] for this CTA's requests

    if (has_rows && tid == 0) {
        // given scores: two arrivals per phase, the cache rows' and the scores'
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], C::GS ? 2 : 1);
            cnt[s] = 0;
        }
        fence_barrier_init();
        cur->b = b0;
        cur->start = start0;
        cur->done = 0;
        cur->issued = 0;
        cur->page_key = pl[2];
        cur->page_id = pl[3];
        cursor_begin_segment<C>(cur, off, end);
        // the ring is untouched: no generic-proxy access precedes these copies;
        // in a decode step the tiles that hold the step's new rows wait
        for (int s = 0; s < C::STAGES; ++s)
            if (!issue_next<C>(cur, P, M, off, smem, full, okf, end, false, C::GS ? pend : nullptr,
                               true))
                break;
    }
    __syncthreads();
    if (local) pdl_wait();  // the private queries (or the scores) come from the previous kernel
    if (has_rows && P.step_rows && tid == 0)  // the tiles held back above (their rows are written)
        while (!cur->done && cur->issued < C::STAGES) issue_next<C>(cur, P, M, off, smem, full, okf, end, false);
    if (has_rows && C::GS && tid == 0)  // the first tiles' score copies
        for (int k = 0; k < cur->issued; ++k)
            issue_scores<C>(smem + (k % C::STAGES) * C::STAGE, M, pend[k % C::STAGES],
                            &full[k % C::STAGES]);
    pdl_launch_dependents();
    if (has_rows) stream_range<C>(M, P, rg, smem);
    // every partial state of this CTA is written: count the CTA, then merge
    // the (request, head) pairs that fall to it once every CTA is counted
    __threadfence();
    __syncthreads();
    if (tid == 0) atomicAdd(ws.cnt, 1);
    merge_phase<C>(P, rg, off, warp, lane, reinterpret_cast<float *>(smem));
}

// The tiles of a CTA's range: scores, online softmax, value reductions; one
// partial state per (request, CTA) segment.
template <class C>
__device__ __forceinline__ void stream_range(const FastMaps &M, const FastParams &P, const CtaRange &rg,
                                             uint8_t *smem) {
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    int *cnt = reinterpret_cast<int *>(smem + C::OFF_CNT);
    int *okf = reinterpret_cast<int *>(smem + C::OFF_OK);
    IssueCursor *cur = reinterpret_cast<IssueCursor *>(smem + C::OFF_CUR);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x;
    const DecodeWs &ws = P.ws;
    const int32_t start0 = rg.start, end = rg.end;
    const int b0 = rg.b0;
    const int32_t *off = rg.off;
    const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
    const int hl = lane >> 4, j = lane & 15;  // this lane's (head slot, tile row)
    // first 16-byte chunk of the shared group of this warp's heads
    const int sgc = (warp * C::HPW) / (C::H / C::NGRP) * C::GCH;
    int hd[C::NH];                            // heads of this lane's slots
#pragma unroll
    for (int i = 0; i < C::NH; ++i) hd[i] = warp * C::HPW + hl + 2 * i;

    float accS[8][4], accR[C::KSP][4];
    float m[C::NH], l[C::NH];
    uint32_t qb[8][2];            // Q^T fragments (shared scores)
    // blockdiag(p)^T fragments: hi and lo bf16 halves, or one f16 (8-bit cache)
    uint32_t pbh[C::KSP][2], pbl[C::Q8 ? 1 : C::KSP][2];
    float fS[2] = {1.f, 1.f}, fR[2] = {1.f, 1.f};  // 8-bit cache: score factors of columns 2tq, 2tq+1
    bool timed_out = false;

    uint32_t it = 0;
    int b = b0;
    int32_t start = start0;
    while (start < end && !timed_out) {
        while (off[b + 1] <= start) ++b;
        const int32_t base = off[b];
        const int32_t seg_end = min(end, off[b + 1]);
        const int t_a = start - base, t_b = seg_end - base;

        // -------- segment set-up: query fragments, private-query fragments, state
#pragma unroll
        for (int i = 0; i < C::NH; ++i) {
            m[i] = -INFINITY;
            l[i] = 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) accS[mt][e] = 0.f;
#pragma unroll
        for (int mt = 0; mt < C::KSP; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) accR[mt][e] = 0.f;
        if constexpr (C::GS) {
            // the scores arrive with the tiles
        } else if constexpr (C::Q8) {
            q8_segment_setup<C>(P, b, warp, gq, tq, qb, pbh, fS, fR,
                                ws.p + ((size_t)b * C::H + warp * C::HPW) * C::R);
        } else {
            // B fragments of Q^T: column n = head warp*HPW + n (n < HPW), else 0
            const bool own = gq < C::HPW;
            const __nv_bfloat16 *qrow = P.q + ((size_t)b * C::H + warp * C::HPW + (own ? gq : 0)) * C::DH;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qb[ks][0] = own ? ld_u32(qrow + ks * 16 + 2 * tq) : 0u;
                qb[ks][1] = own ? ld_u32(qrow + ks * 16 + 2 * tq + 8) : 0u;
            }
            // B fragments of blockdiag(p)^T over the warp's HPW*R private
            // columns: entry (k, n) is p[head n][k - n R] when k falls in head
            // n's columns, else 0
            const float *pw = ws.p + ((size_t)b * C::H + warp * C::HPW) * C::R;
#pragma unroll
            for (int ks = 0; ks < C::KSP; ++ks) {
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k = ks * 16 + 2 * tq + (e & 1) + (e >> 1) * 8;
                    v[e] = (own && k / C::R == gq) ? pw[k] : 0.f;  // pw[k] = p[head k/R][k%R]
                }
                float hv[4], lv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    hv[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
                    lv[e] = v[e] - hv[e];
                }
                pbh[ks][0] = pack_bf16(hv[0], hv[1]);
                pbh[ks][1] = pack_bf16(hv[2], hv[3]);
                pbl[ks][0] = pack_bf16(lv[0], lv[1]);
                pbl[ks][1] = pack_bf16(lv[2], lv[3]);
            }
        }

        // -------- stream the segment's tiles
        for (int t = t_a / C::TS * C::TS; t < t_b; t += C::TS, ++it) {
            const int s = it % C::STAGES;
            if (!mbar_wait(&full[s], (it / C::STAGES) & 1)) {
                if (lane == 0) status_or(P.status, LRKV_STATUS_TIMEOUT);
                timed_out = true;
                break;
            }
            const bool page_ok = okf[s] != 0;
            const uint8_t *st = smem + s * C::STAGE;
            const int mi = lane >> 3;
#pragma unroll
            for (int h2 = 0; h2 < C::TS / 16; ++h2) {  // 16-row halves of the stage
            const int t16 = t + 16 * h2;                 // first row of this half
            const bool partial = !page_ok || t16 < t_a || t16 + 16 > t_b;
            const bool valid = page_ok && t16 + j >= t_a && t16 + j < t_b;

            // scores: D[row x head] = S_K . Q^T + R_K(warp columns) . blockdiag(p)^T,
            // accumulated in four independent chains (shared even/odd k-steps,
            // private hi/lo halves) so the tensor-core latency overlaps
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (C::GS) {
                // given scores: read per lane in the softmax below
            } else if constexpr (C::Q8) {
                q8_scores<C>(st, 16 * h2, warp, gq, tq, qb, pbh, fS, fR, c);
            } else {
                float c1[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
                float c3[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t skb = smem_u32(st + C::OFF_SK);
                const uint32_t rkb = smem_u32(st + C::OFF_RK);
                const int rr = (mi & 1) * 8 + (lane & 7);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a[4];
                    ldmatrix_x4(skb + box_chunk_rows<C::TS>(16 * h2 + rr, sgc + 2 * ks + (mi >> 1)), a[0], a[1], a[2], a[3]);
                    if (ks & 1) mma_bf16_16816(c1, a, qb[ks][0], qb[ks][1]);
                    else mma_bf16_16816(c, a, qb[ks][0], qb[ks][1]);
                }
                const int cw = warp * (C::HPW * C::R / 8);  // first 16-byte chunk of the warp's columns
#pragma unroll
                for (int ks = 0; ks < C::KSP; ++ks) {
                    uint32_t a[4];
                    ldmatrix_x4(rkb + box_chunk_rows<C::TS>(16 * h2 + rr, cw + 2 * ks + (mi >> 1)), a[0], a[1], a[2], a[3]);
                    mma_bf16_16816(c2, a, pbh[ks][0], pbh[ks][1]);
                    mma_bf16_16816(c3, a, pbl[ks][0], pbl[ks][1]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) c[e] = (c[e] + c1[e]) + (c2[e] + c3[e]);
            }

            // softmax per (head slot, row) lane; lazy reference maximum
            float pe[C::NH], al[C::NH];
            bool rescale = false;
#pragma unroll
            for (int i = 0; i < C::NH; ++i) {
                float sc;
                if constexpr (C::GS) {
                    sc = valid ? reinterpret_cast<const float *>(st + C::OFF_SC)[(16 * h2 + j) * C::H + hd[i]] *
                                     P.scale_log2
                               : -INFINITY;
                } else {
                    // D[row j][head n = hl + 2i] sits in lane (j % 8) * 4 + i, register hl + 2 (j / 8)
                    const int src = (j & 7) * 4 + i;
                    const float v0 = __shfl_sync(0xffffffffu, c[0], src);
                    const float v1 = __shfl_sync(0xffffffffu, c[1], src);
                    const float v2 = __shfl_sync(0xffffffffu, c[2], src);
                    const float v3 = __shfl_sync(0xffffffffu, c[3], src);
                    const float lo = hl ? v1 : v0, hi = hl ? v3 : v2;
                    sc = valid ? ((j < 8) ? lo : hi) * P.scale_log2 : -INFINITY;
                }
                if (P.norm && valid)  // joint key norm of (row j, head hd[i])
                    sc *= __bfloat162float(
                        reinterpret_cast<const __nv_bfloat16 *>(st + C::OFF_NK)[(16 * h2 + j) * C::H + hd[i]]);
                float mx = sc;
#pragma unroll
                for (int o = 8; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_old = m[i];
                const float m_new = (mx > m_old + kLazyMax) ? mx : m_old;
                const float alpha = (m_new == m_old) ? 1.f : exp2f(m_old - m_new);
                const float e = (valid && m_new != -INFINITY) ? exp2f(sc - m_new) : 0.f;
                float sum = e;
#pragma unroll
                for (int o = 8; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                l[i] = l[i] * alpha + sum;
                m[i] = m_new;
                pe[i] = e;
                al[i] = alpha;
                rescale |= alpha != 1.f;
            }

            // values: accS += S_V^T . P^T, accR += R_V^T(warp columns) . P^T
            {
                // B fragment: column n = gq (< HPW) holds P of head slot (n & 1, n >> 1)
                // at rows 2tq, 2tq+1 and 2tq+8, 2tq+9
                const int sl = (gq & 1) * 16 + 2 * tq;
                float w0 = 0.f, w1 = 0.f, w8 = 0.f, w9 = 0.f;
#pragma unroll
                for (int i = 0; i < C::NH; ++i) {
                    const float x0 = __shfl_sync(0xffffffffu, pe[i], sl);
                    const float x1 = __shfl_sync(0xffffffffu, pe[i], sl + 1);
                    const float x8 = __shfl_sync(0xffffffffu, pe[i], sl + 8);
                    const float x9 = __shfl_sync(0xffffffffu, pe[i], sl + 9);
                    if ((gq >> 1) == i) { w0 = x0; w1 = x1; w8 = x8; w9 = x9; }
                }
                if (gq >= C::HPW) w0 = w1 = w8 = w9 = 0.f;
                // 8-bit cache: one f16 per weight (11 significant bits)
                const uint32_t fh0 = C::Q8 ? pack_f16(w0, w1) : 0u, fh1 = C::Q8 ? pack_f16(w8, w9) : 0u;
                const __nv_bfloat16 h0 = __float2bfloat16_rn(w0), h1 = __float2bfloat16_rn(w1);
                const __nv_bfloat16 h8 = __float2bfloat16_rn(w8), h9 = __float2bfloat16_rn(w9);
                const uint32_t bh0 = pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
                const uint32_t bh1 = pack_bf16(__bfloat162float(h8), __bfloat162float(h9));
                const uint32_t bl0 = pack_bf16(w0 - __bfloat162float(h0), w1 - __bfloat162float(h1));
                const uint32_t bl1 = pack_bf16(w8 - __bfloat162float(h8), w9 - __bfloat162float(h9));
                if (__any_sync(0xffffffffu, rescale)) {
                    // factors of columns 2tq and 2tq+1 (head slot tq of lanes 0 and 16)
                    float a0 = 1.f, a1 = 1.f;
#pragma unroll
                    for (int i = 0; i < C::NH; ++i) {
                        const float y0 = __shfl_sync(0xffffffffu, al[i], 0);
                        const float y1 = __shfl_sync(0xffffffffu, al[i], 16);
                        if (tq == i) { a0 = y0; a1 = y1; }
                    }
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        accS[mt][0] *= a0; accS[mt][1] *= a1;
                        accS[mt][2] *= a0; accS[mt][3] *= a1;
                    }
#pragma unroll
                    for (int mt = 0; mt < C::KSP; ++mt) {
                        accR[mt][0] *= a0; accR[mt][1] *= a1;
                        accR[mt][2] *= a0; accR[mt][3] *= a1;
                    }
                }
                uint32_t m01 = 0xffffffffu, m89 = 0xffffffffu;
                if (partial) {
                    auto ok = [&](int r) { return page_ok && t16 + r >= t_a && t16 + r < t_b; };
                    m01 = (ok(2 * tq) ? 0x0000ffffu : 0u) | (ok(2 * tq + 1) ? 0xffff0000u : 0u);
                    m89 = (ok(2 * tq + 8) ? 0x0000ffffu : 0u) | (ok(2 * tq + 9) ? 0xffff0000u : 0u);
                }
                if constexpr (C::Q8) {
                    if (partial) q8_values<C, true>(st, 16 * h2, warp, gq, tq, m01, m89, fh0, fh1, accS, accR);
                    else q8_values<C, false>(st, 16 * h2, warp, gq, tq, m01, m89, fh0, fh1, accS, accR);
                } else {
                const int rr = (mi >> 1) * 8 + (lane & 7);
                const uint32_t svb = smem_u32(st + C::OFF_SV);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    uint32_t a[4];
                    ldmatrix_x4_trans(svb + box_chunk_rows<C::TS>(16 * h2 + rr, sgc + 2 * mt + (mi & 1)), a[0], a[1], a[2], a[3]);
                    a[0] &= m01; a[1] &= m01; a[2] &= m89; a[3] &= m89;
                    mma_bf16_16816(accS[mt], a, bh0, bh1);
                    mma_bf16_16816(accS[mt], a, bl0, bl1);
                }
                const uint32_t rvb = smem_u32(st + C::OFF_RV);
                const int cw = warp * (C::HPW * C::R / 8);
#pragma unroll
                for (int mt = 0; mt < C::KSP; ++mt) {
                    uint32_t a[4];
                    ldmatrix_x4_trans(rvb + box_chunk_rows<C::TS>(16 * h2 + rr, cw + 2 * mt + (mi & 1)), a[0], a[1], a[2], a[3]);
                    a[0] &= m01; a[1] &= m01; a[2] &= m89; a[3] &= m89;
                    mma_bf16_16816(accR[mt], a, bh0, bh1);
                    mma_bf16_16816(accR[mt], a, bl0, bl1);
                }
                }
            }

            }  // halves

            // release the stage; the last warp out refills it
            __syncwarp();
            if (lane == 0) {
                int prev;
                asm volatile("atom.acq_rel.cta.shared::cta.add.s32 %0, [%1], 1;"
                             : "=r"(prev)
                             : "r"(smem_u32(&cnt[s]))
                             : "memory");
                if (prev == C::NCW - 1) {
                    cnt[s] = 0;
                    issue_next<C>(cur, P, M, off, smem, full, okf, end);
                }
            }
            __syncwarp();
        }
        // -------- segment end: this warp's heads of partial slot b + g
        const size_t slot = (size_t)b + g;
        const size_t W = C::DH + C::R;
        if (!timed_out) {  // (a timed-out warp leaves its partial unwritten)
#pragma unroll
        for (int i = 0; i < C::NH; ++i) {
            if (j == 0) {
                ws.ml[(slot * C::H + hd[i]) * 2 + 0] = m[i];
                ws.ml[(slot * C::H + hd[i]) * 2 + 1] = l[i];
            }
        }
        if constexpr (C::Q8) {
            q8_write_partial<C>(P, slot, warp, gq, tq, accS, accR);
        } else {
        if (2 * tq < C::HPW) {
            const int h0 = warp * C::HPW + 2 * tq;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int d = mt * 16 + gq;
                ws.acc[(slot * C::H + h0) * W + d] = accS[mt][0];
                ws.acc[(slot * C::H + h0 + 1) * W + d] = accS[mt][1];
                ws.acc[(slot * C::H + h0) * W + d + 8] = accS[mt][2];
                ws.acc[(slot * C::H + h0 + 1) * W + d + 8] = accS[mt][3];
            }
        }
        // private reduction: accumulator row mm (a private column of the
        // warp) is useful in column n = mm / R (its own head)
#pragma unroll
        for (int mt = 0; mt < C::KSP; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int mm = mt * 16 + gq + (e >> 1) * 8;
                const int n = 2 * tq + (e & 1);
                if (n < C::HPW && mm / C::R == n)
                    ws.acc[(slot * C::H + warp * C::HPW + n) * W + C::DH + (mm - n * C::R)] = accR[mt][e];
            }
        }
        }  // !timed_out
        if (timed_out) break;
        start = seg_end;
    }

    // Never leave with copies in flight into this CTA's shared memory (only
    // possible after a timeout: normally every issued tile was consumed).
    __syncthreads();
    if (tid == 0) {
        const int issued = cur->issued;
        for (int k = (int)it; k < issued; ++k) mbar_wait(&full[k % C::STAGES], (k / C::STAGES) & 1);
    }
}

// ---------------------------------------------------------------------------
// Merge of a request's segment states into its output (section 3 after
// Algorithm 2: one softmax over the whole sequence -- the segments' (m, l,
// accS, accR) combine by the log-sum-exp rule -- and equation 7's expansion
// by B_V[h], once, on the merged private accumulator):
//     out[b, h] = accS / L + (accR / L) B_V[h]^T.
// A (request, head) pair is merged by WP warps of one CTA: warp k of the
// group takes segments k, k + WP, ... and keeps a running (M, L, acc) over
// batches of eight segments whose loads are all in flight; lane i holds value
// columns 2i, 2i + 1 and 64 + 2i, 65 + 2i of accS and, for 2i < r, columns
// 2i, 2i + 1 of accR.  The group's first warp then combines the WP states in
// warp order through shared memory and expands.  Partial states come from L2
// (other CTAs wrote them).
// ---------------------------------------------------------------------------
struct MergeState {
    float M, L;
    float2 a0, a1, ar;
};

template <class C>
__device__ __forceinline__ MergeState merge_segments(const FastParams &P, size_t s0, int first,
                                                     int step, int nseg, int lane) {
    constexpr int W = C::DH + C::R, U = 8;
    const bool has_r = 2 * lane < C::R;
    MergeState st{-INFINITY, 0.f, make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    for (int s = first; s < nseg; s += U * step) {
        float2 ml[U], v0[U], v1[U], vr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            ml[u] = make_float2(-INFINITY, 0.f);
            v0[u] = v1[u] = vr[u] = make_float2(0.f, 0.f);
            if (s + u * step < nseg) {
                const size_t slot = s0 + (size_t)(s + u * step) * C::H;
                const float *acc = P.ws.acc + slot * W;
                ml[u] = __ldcg(reinterpret_cast<const float2 *>(P.ws.ml + slot * 2));
                v0[u] = __ldcg(reinterpret_cast<const float2 *>(acc + 2 * lane));
                v1[u] = __ldcg(reinterpret_cast<const float2 *>(acc + 64 + 2 * lane));
                if (has_r) vr[u] = __ldcg(reinterpret_cast<const float2 *>(acc + C::DH + 2 * lane));
            }
        }
        float Mb = st.M;
#pragma unroll
        for (int u = 0; u < U; ++u) Mb = fmaxf(Mb, ml[u].x);
        if (Mb == -INFINITY) continue;  // nothing visible so far
        const float sc = st.M == -INFINITY ? 0.f : exp2f(st.M - Mb);
        st.L *= sc;
        st.a0.x *= sc; st.a0.y *= sc; st.a1.x *= sc; st.a1.y *= sc; st.ar.x *= sc; st.ar.y *= sc;
        st.M = Mb;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float w = (ml[u].x == -INFINITY) ? 0.f : exp2f(ml[u].x - Mb);
            st.L = fmaf(w, ml[u].y, st.L);
            st.a0.x = fmaf(w, v0[u].x, st.a0.x); st.a0.y = fmaf(w, v0[u].y, st.a0.y);
            st.a1.x = fmaf(w, v1[u].x, st.a1.x); st.a1.y = fmaf(w, v1[u].y, st.a1.y);
            st.ar.x = fmaf(w, vr[u].x, st.ar.x); st.ar.y = fmaf(w, vr[u].y, st.ar.y);
        }
    }
    return st;
}

// Expansion and store of a merged state: out[b, h] = a / L + (ar / L) B_V[h]^T
// (bvr: this lane's four B_V rows, loaded beforehand).
template <class C>
__device__ __forceinline__ void merge_store(const FastParams &P, int b, int h, const MergeState &st,
                                            const uint4 (&bvr)[4][C::R / 8], int lane) {
    const float inv = st.L > 0.f ? 1.f / st.L : 0.f;
    float o[4] = {st.a0.x * inv, st.a0.y * inv, st.a1.x * inv, st.a1.y * inv};
#pragma unroll
    for (int k = 0; k < C::R / 8; ++k) {
        float r[8];  // (accR / L)[8k .. 8k + 7], from lanes 4k .. 4k + 3
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            r[2 * e] = __shfl_sync(0xffffffffu, st.ar.x, 4 * k + e) * inv;
            r[2 * e + 1] = __shfl_sync(0xffffffffu, st.ar.y, 4 * k + e) * inv;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t wd = u4w(bvr[i][k], e);
                o[i] = fmaf(r[2 * e], bf16_lo(wd), o[i]);
                o[i] = fmaf(r[2 * e + 1], bf16_hi(wd), o[i]);
            }
    }
    __nv_bfloat16 *dst = P.out + ((size_t)b * C::H + h) * C::DH;
    *reinterpret_cast<uint32_t *>(dst + 2 * lane) = pack_bf16(o[0], o[1]);
    *reinterpret_cast<uint32_t *>(dst + 64 + 2 * lane) = pack_bf16(o[2], o[3]);
}

// The grid's last phase.  Once every CTA has written its partial states
// (the workspace counter reaches the grid size; a bounded wait), CTA g merges the
// (request, head) pairs g, g + G, ...: in rounds of up to eight pairs, each
// pair on WP = 8 / (pairs in the round) warps (a power of two).  A request
// of invalid length has no segment; its zero output was written by the
// kernel that started the decode.  Offsets: the CTA's full table (batches of
// at most kLocalReq requests) or the prologue's.  `scratch`: 8 KB of shared
// memory no longer in use (the first ring stage).
template <class C>
__device__ void merge_phase(const FastParams &P, const CtaRange &rg, const int32_t *off, int warp,
                            int lane, float *scratch) {
    constexpr int NO = C::R / 8;
    const int32_t *full_off = P.B <= kLocalReq ? off : P.ws.off;
    const int npairs = P.B * C::H, G = (int)gridDim.x, g = blockIdx.x;
    const int mine = npairs > g ? (npairs - g + G - 1) / G : 0;  // pairs of this CTA
    if (mine == 0) return;
    for (int r0 = 0; r0 < mine; r0 += C::NCW) {
        const int nr = min(C::NCW, mine - r0);
        const int wp = nr > 4 ? 1 : nr > 2 ? 2 : nr > 1 ? 4 : 8;  // warps per pair
        const int slot = warp / wp, part = warp % wp;
        const bool active = slot < nr;
        int b = 0, h = 0, g_lo = 0, nseg = 0;
        if (active) {
            const int i = g + (r0 + slot) * G;
            b = i / C::H;
            h = i % C::H;
            const int32_t o0 = full_off[b], o1 = full_off[b + 1];
            if (o1 > o0) {
                g_lo = o0 / rg.chunk;
                nseg = (o1 - 1) / rg.chunk - g_lo + 1;
            }
        }
        // the expanding warp's B_V rows, in flight across the wait
        uint4 bvr[4][NO];
        if (active && part == 0 && nseg > 0) {
            const __nv_bfloat16 *bv = P.B_V + (size_t)h * C::DH * C::R;
            const int dd[4] = {2 * lane, 2 * lane + 1, 64 + 2 * lane, 65 + 2 * lane};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int k = 0; k < NO; ++k)
                    bvr[i][k] = __ldg(reinterpret_cast<const uint4 *>(bv + (size_t)dd[i] * C::R + 8 * k));
        }
        if (r0 == 0) wait_grid_count(P);  // (flagged on timeout; merges stale states)
        MergeState st{-INFINITY, 0.f, make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        if (active && nseg > 0)
            st = merge_segments<C>(P, (size_t)(b + g_lo) * C::H + h, part, wp, nseg, lane);
        if (wp > 1) {
            // [warp][lane][8]: M, L, a0, a1, ar
            float *my = scratch + (warp * 32 + lane) * 8;
            reinterpret_cast<float4 *>(my)[0] = make_float4(st.M, st.L, st.a0.x, st.a0.y);
            reinterpret_cast<float4 *>(my)[1] = make_float4(st.a1.x, st.a1.y, st.ar.x, st.ar.y);
            __syncthreads();
            if (active && part == 0 && nseg > 0) {
                float M = st.M;
                for (int k = 1; k < wp; ++k) M = fmaxf(M, scratch[((warp + k) * 32 + lane) * 8]);
                MergeState t{M, 0.f, make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                if (M != -INFINITY)
                    for (int k = 0; k < wp; ++k) {
                        const float *o = scratch + ((warp + k) * 32 + lane) * 8;
                        const float w = o[0] == -INFINITY ? 0.f : exp2f(o[0] - M);
                        t.L = fmaf(w, o[1], t.L);
                        t.a0.x = fmaf(w, o[2], t.a0.x); t.a0.y = fmaf(w, o[3], t.a0.y);
                        t.a1.x = fmaf(w, o[4], t.a1.x); t.a1.y = fmaf(w, o[5], t.a1.y);
                        t.ar.x = fmaf(w, o[6], t.ar.x); t.ar.y = fmaf(w, o[7], t.ar.y);
                    }
                st = t;
            }
            __syncthreads();  // the scratch is reused by the next round
        }
        if (active && part == 0 && nseg > 0) merge_store<C>(P, b, h, st, bvr, lane);
    }
}

// ---------------------------------------------------------------------------
// Rotary scores (reading note, section 8: exact RoPE over the factored
// cache) for bf16 caches with d_h = 128, on 5th-generation tensor cores.
//
// With i the query's position, q~ = q D_i and j a key's position, the score
// of head h is
//     q~ . (S_K[j] D_j)  +  (C_j W_h) . R_K[h, j]
// where C_j is the key's (cos, sin)(j theta_c) table row, interleaved by
// channel pair, and W_h = [A; Bq] (d_h x r) comes from the prologue (see
// rope_fast_operands): D_{i-j} = D_i D_j^T turns the note's per-distance
// private query (q D_{i-j}) B_K[h] into a product of a row that depends only
// on j and a matrix that depends only on the step.  The kernel writes the raw
// score of every visible (row, head) to the plan-ordered score array; the
// split kernel's given-score mode then streams S_V, R_V and those scores.
//
// A CTA takes a range of rows (the split kernel's plan, one range per NG
// CTAs) for a group of g heads (g = rope_tc_heads_per_cta(r)), in 128-row
// tiles of one request:
//   * warp 0 (one thread) lands by TMA, per tile, the table rows (f16) and
//     the S_K rows (bf16) as two K-halves of 64 channels through a ring of
//     half-tile stages (128-byte swizzle), and the group's R_K columns
//     (bf16, 128- or 64-byte swizzle) into a ring of tile buffers; the S_K and
//     R_K rows come in pieces of 32 to 128 rows, each inside one page.  Per
//     request it lands the group's W^T (f16, [g r][128]) and query block
//     (bf16, [16][128]);
//   * warps 2-9 turn each landed S_K channel pair by its table entry in
//     place (fp32, rounded to bf16);
//   * warp 1 (one thread) issues tcgen05.mma (kind::f16, M = 128, fp32
//     accumulate in tensor memory): the private products C_tile . W (N = g r)
//     and the shared term (turned S_K) . [q~ values; q~ remainders]^T
//     (N = 16), into one of two 256-column accumulators;
//   * one tile later, warps 2-9 read the accumulator back (tcgen05.ld, one
//     tile row per thread; two warps share a 32-lane quarter, each for half
//     the heads), dot each head's r private columns with the row's R_K[h]
//     from shared memory (the swizzle makes the row-per-thread reads free of
//     bank conflicts), scale by the inverse W scale, add the shared value and
//     remainder, and store the row's scores.
// ---------------------------------------------------------------------------
template <int H_, int R_>
struct RtcCfg {
    static constexpr int H = H_, R = R_, DH = 128, TM = 128;  // tile rows = MMA M
    static constexpr int HPC = rope_tc_heads_per_cta(R);       // heads per CTA
    static constexpr int NG = H / HPC;                          // CTAs per row range
    static constexpr int NPRIV = HPC * R;                       // private MMA N
    static constexpr int EPI = 8, NT = (2 + EPI) * 32;          // producer, MMA, 8 turn/epilogue warps
    static constexpr int HPE = HPC / 2;                         // heads per epilogue warp
    static constexpr int HALF = TM * 128;                       // one K-half of a tile: 16 KB
    static constexpr int STAGE = 2 * HALF;                      // half-tile stage: table + S_K
    // R_K columns of the group: blocks of SWZ bytes per row (128-byte swizzle
    // when the group's columns fill 64-element blocks, else 64-byte)
    static constexpr int SWZ = (NPRIV % 64 == 0) ? 128 : 64;
    static constexpr int RBLK = SWZ / 2;                        // elements per block row
    static constexpr int NRB = NPRIV / RBLK;                    // blocks
    static constexpr int RK_TILE = NRB * TM * SWZ;              // = TM * NPRIV * 2 bytes
    static constexpr int W_BYTES = 2 * NPRIV * 128;             // W^T of the group, two K-halves
    static constexpr int QB_BYTES = 2 * 16 * 128;               // query block, two K-halves
    // two R_K buffers when that leaves two tiles of stages, up to four stages
    static constexpr int BUDGET = 227 * 1024 - 3072 - W_BYTES - QB_BYTES;
    static constexpr int RKB = (BUDGET - 2 * RK_TILE) / STAGE >= 2 ? 2 : 1;
    static constexpr int S_FIT = (BUDGET - RKB * RK_TILE) / STAGE;
    static constexpr int STAGES = S_FIT > 4 ? 4 : S_FIT;
    static constexpr int OFF_RK = STAGES * STAGE;
    static constexpr int OFF_W = OFF_RK + RKB * RK_TILE;
    static constexpr int OFF_QB = OFF_W + W_BYTES;
    // full[S], turned[S], empty[S], wfull, wfree, rkfull[2], rkfree[2],
    // acc_full[2], acc_empty[2], drain
    static constexpr int OFF_BAR = OFF_QB + QB_BYTES;
    static constexpr int OFF_TMEM = OFF_BAR + 8 * (3 * STAGES + 11);
    static constexpr int OFF_PLAN = OFF_TMEM + 16;
    static constexpr int SMEM = OFF_PLAN + 512 + 1024;  // + alignment slack
    static constexpr int ACC = 256, SH_COL = 224;       // accumulator a at 256 a; shared term at +224
    static constexpr uint32_t TMEM_COLS = 512;

    static_assert(H % HPC == 0 && HPC % 2 == 0, "whole head groups, two epilogue halves");
    static_assert(STAGES >= 2, "a tile's two halves in flight");
    static_assert(NPRIV <= SH_COL && NPRIV % 32 == 0, "private N fits before the shared columns");
    static_assert((HPE * R) % 16 == 0, "whole 16-column TMEM loads per epilogue warp");
    static_assert(W_BYTES % 1024 == 0 && RK_TILE % 1024 == 0, "1 KB-aligned swizzled buffers");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct RtcMaps {
    CUtensorMap tab, sk, rk, wt, qb;
};

// The 128-row tiles of a CTA's range in order: request segments, tiles
// aligned to the request's positions.
struct TileWalk {
    int b, seg;
    int32_t base, t, t_a, t_b, start;
    bool done;
};

__device__ __forceinline__ void walk_segment(TileWalk &w, const int32_t *off, int32_t end, int tm) {
    while (off[w.b + 1] <= w.start) ++w.b;
    w.base = off[w.b];
    w.t_a = w.start - w.base;
    w.t_b = min(end, off[w.b + 1]) - w.base;
    w.t = w.t_a / tm * tm;
}

__device__ __forceinline__ TileWalk walk_begin(const CtaRange &rg, int tm) {
    TileWalk w;
    w.b = rg.b0;
    w.seg = 0;
    w.start = rg.start;
    w.done = rg.start >= rg.end;
    if (!w.done) walk_segment(w, rg.off, rg.end, tm);
    return w;
}

__device__ __forceinline__ void walk_next(TileWalk &w, const CtaRange &rg, int tm) {
    w.t += tm;
    if (w.t >= w.t_b) {
        w.start = w.base + w.t_b;
        if (w.start >= rg.end) {
            w.done = true;
            return;
        }
        ++w.seg;
        walk_segment(w, rg.off, rg.end, tm);
    }
}

// A bf16 channel pair (2c, 2c+1) turned by its f16 (cos, sin) table entry.
__device__ __forceinline__ uint32_t turn_pair(uint32_t s, uint32_t cs) {
    const float x0 = bf16lo(s), x1 = bf16hi(s);
    const float2 r = __half22float2(*reinterpret_cast<const __half2 *>(&cs));
    return pack_bf16(x0 * r.x - x1 * r.y, x0 * r.y + x1 * r.x);
}

__device__ __forceinline__ uint32_t u4_word(const uint4 &v, int w) {
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

template <class C>
__global__ void __launch_bounds__(C::NT, 1)
    rope_scores_tc_kernel(const __grid_constant__ RtcMaps M, const FastParams P, int br) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *turned = full + C::STAGES;
    uint64_t *empty = turned + C::STAGES;
    uint64_t *wfull = empty + C::STAGES;
    uint64_t *wfree = wfull + 1;
    uint64_t *rkfull = wfree + 1;
    uint64_t *rkfree = rkfull + 2;
    uint64_t *acc_full = rkfree + 2;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM);
    int32_t *pl = reinterpret_cast<int32_t *>(smem + C::OFF_PLAN);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = blockIdx.x % C::NG;
    if (tid == 32) {
        prefetch_tensormap(&M.tab);
        prefetch_tensormap(&M.sk);
        prefetch_tensormap(&M.rk);
        prefetch_tensormap(&M.wt);
        prefetch_tensormap(&M.qb);
    }
    if (!P.req_row) {  // the producer reads the page-table rows right after the plan
        const size_t pt_bytes = (size_t)P.B * P.max_pages * sizeof(int32_t);
        if (pt_bytes <= 64 * 1024)
            for (size_t o = (size_t)tid * 128; o < pt_bytes; o += (size_t)C::NT * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(P.page_table) + o));
    }
    const CtaRange rg = cta_range<C::NT>(P, blockIdx.x / C::NG, gridDim.x / C::NG, pl);
    if (rg.start >= rg.end) {
        pdl_wait();
        return;
    }
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&turned[s], C::EPI);
            mbar_init(&empty[s], 1);
        }
        mbar_init(wfull, 1);
        mbar_init(wfree, 1);
        for (int k = 0; k < 2; ++k) {
            mbar_init(&rkfull[k], 1);
            mbar_init(&rkfree[k], C::EPI);
            mbar_init(&acc_full[k], 1);
            mbar_init(&acc_empty[k], C::EPI);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // W, the query blocks and their scales come from the prologue
    pdl_wait();
    pdl_launch_dependents();
    bool ok = true;

    if (warp == 0 && lane == 0) {
        // ---- producer
        TileWalk w = walk_begin(rg, C::TM);
        int it = 0, i = 0, seg_loaded = -1;
        // page ids of a tile's pieces (br rows, inside one page), read one
        // tile ahead so that their latency passes while the producer waits
        int32_t pid[C::TM / 32];
        int np = 0;
        auto read_pages = [&](const TileWalk &tw) {
            const int32_t *pt = page_row(P, tw.b);
            np = 0;
#pragma unroll
            for (int p = 0; p < C::TM / 32; ++p) {
                const int pos = tw.t + p * br;
                if (p < C::TM / br && pos < tw.t_b) {
                    pid[p] = pt[pos / P.page_size];
                    np = p + 1;
                }
            }
        };
        if (!w.done) read_pages(w);
        while (!w.done) {
            if (w.seg != seg_loaded) {
                // the previous request's products are done with W
                if (seg_loaded >= 0 && !mbar_wait(wfree, seg_loaded & 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(wfull, C::W_BYTES + C::QB_BYTES);
                tma_load_3d(smem + C::OFF_W, &M.wt, 0, (w.b * C::H + grp * C::HPC) * C::R, 0, wfull);
                tma_load_3d(smem + C::OFF_QB, &M.qb, 0, (w.b * C::NG + grp) * 16, 0, wfull);
                seg_loaded = w.seg;
            }
            int prow[C::TM / 32];
            for (int kh = 0; kh < 2; ++kh, ++it) {
                const int s = it % C::STAGES;
                if (it >= C::STAGES && !mbar_wait(&empty[s], ((it / C::STAGES) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (kh == 0) {
                    // pool rows of the pieces; pieces past the segment's end are
                    // not loaded (their rows are not stored)
#pragma unroll
                    for (int p = 0; p < C::TM / 32; ++p) {
                        if (p >= np) continue;
                        int32_t page = pid[p];
                        if (page < 0 || page >= P.num_pages) {
                            status_or(P.status, LRKV_STATUS_BAD_PAGE);
                            page = 0;
                        }
                        prow[p] = page * P.page_size + (w.t + p * br) % P.page_size;
                    }
                }
                uint8_t *st = smem + s * C::STAGE;
                mbar_arrive_expect_tx(&full[s], C::HALF + np * br * 128);
                tma_load_3d(st, &M.tab, 0, w.t, kh, &full[s]);
#pragma unroll
                for (int p = 0; p < C::TM / 32; ++p)
                    if (p < np) tma_load_3d(st + C::HALF + p * br * 128, &M.sk, 0, prow[p], kh, &full[s]);
            }
            if (!ok) break;
            // the tile's R_K columns of the group (read once: evict first)
            const int rb = i % C::RKB;
            if (i >= C::RKB && !mbar_wait(&rkfree[rb], ((i / C::RKB) - 1) & 1)) {
                ok = false;
                break;
            }
            uint8_t *rk = smem + C::OFF_RK + rb * C::RK_TILE;
            mbar_arrive_expect_tx(&rkfull[rb], np * br * C::NPRIV * 2);
            const uint64_t ef = l2_evict_first_policy();
#pragma unroll
            for (int p = 0; p < C::TM / 32; ++p)
                if (p < np)
#pragma unroll
                    for (int k = 0; k < C::NRB; ++k)
                        tma_load_3d_hint(rk + k * (C::TM * C::SWZ) + p * br * C::SWZ, &M.rk, 0, prow[p],
                                         grp * C::NRB + k, &rkfull[rb], ef);
            ++i;
            walk_next(w, rg, C::TM);
            if (!w.done) read_pages(w);
        }
        // never leave with copies in flight into this CTA's shared memory
        for (int k = max(0, it - C::STAGES); k < it; ++k)
            mbar_wait(&full[k % C::STAGES], (k / C::STAGES) & 1);
        for (int k = max(0, i - C::RKB); k < i; ++k) mbar_wait(&rkfull[k % C::RKB], (k / C::RKB) & 1);
        if (seg_loaded >= 0) mbar_wait(wfull, seg_loaded & 1);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t id_p = tc_idesc_f16(C::TM, C::NPRIV), id_s = tc_idesc_bf16(C::TM, 16);
        const uint32_t wbase = smem_u32(smem + C::OFF_W), qbase = smem_u32(smem + C::OFF_QB);
        TileWalk w = walk_begin(rg, C::TM);
        int it = 0, i = 0, seg_cur = -1;
        while (!w.done && ok) {
            if (w.seg != seg_cur) {
                if (seg_cur >= 0) tc_commit(wfree);  // W is free once these products read it
                seg_cur = w.seg;
                if (!mbar_wait(wfull, seg_cur & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            const int a = i & 1;
            if (i >= 2 && !mbar_wait(&acc_empty[a], ((i >> 1) - 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t dp = tmem + a * C::ACC, ds = dp + C::SH_COL;
            // private products: C_tile (f16) . W (f16), K = 128 in two halves
            for (int kh = 0; kh < 2 && ok; ++kh) {
                const int k = it + kh, s = k % C::STAGES;
                if (!mbar_wait(&full[s], (k / C::STAGES) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sw128_kmajor_desc(smem_u32(smem + s * C::STAGE));
                const uint64_t bd = sw128_kmajor_desc(wbase + kh * C::NPRIV * 128);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_f16(dp, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), id_p, (kh | kk) != 0);
            }
            // shared term: turned S_K (bf16) . query block (bf16); a half's
            // stage is free once these products have read it
            for (int kh = 0; kh < 2 && ok; ++kh) {
                const int k = it + kh, s = k % C::STAGES;
                if (!mbar_wait(&turned[s], (k / C::STAGES) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sw128_kmajor_desc(smem_u32(smem + s * C::STAGE + C::HALF));
                const uint64_t bd = sw128_kmajor_desc(qbase + kh * 2048);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_f16(ds, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), id_s, (kh | kk) != 0);
                tc_commit(&empty[s]);
            }
            if (!ok) break;
            tc_commit(&acc_full[a]);
            it += 2;
            ++i;
            walk_next(w, rg, C::TM);
        }
        // every issued product has completed before tensor memory is freed
        tc_commit(drain);
        mbar_wait(drain, 0);
    } else if (warp >= 2) {
        // ---- turn S_K, then the epilogue one tile later
        const int ew = warp - 2, q4 = warp & 3, row = 32 * q4 + lane;
        const int hh = ew >> 2;                          // half of the group's heads
        const int h0 = grp * C::HPC + hh * C::HPE;       // this thread's first head
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        TileWalk w = walk_begin(rg, C::TM);
        int it = 0, i = 0, seg_cur = -1;
        float winv[C::HPE];
        struct Pending {
            bool on;
            int i;
            int64_t g;  // score-array row (-1: not stored)
            float winv[C::HPE];
        } pd;
        pd.on = false;
        auto finish = [&](const Pending &q) -> bool {
            const int a = q.i & 1, rb = q.i % C::RKB;
            if (!mbar_wait(&acc_full[a], (q.i >> 1) & 1) || !mbar_wait(&rkfull[rb], (q.i / C::RKB) & 1)) {
                if (lane == 0) status_or(P.status, LRKV_STATUS_TIMEOUT);
                return false;
            }
            tc_fence_after();
            // this row's R_K columns from the swizzled tile: logical 16-byte
            // chunk x of block k sits at chunk x ^ (row bits) of the row
            const uint8_t *rk = smem + C::OFF_RK + rb * C::RK_TILE + row * C::SWZ;
            const int sw = C::SWZ == 128 ? (row & 7) : ((row >> 1) & 3);
            float pr[C::HPE];
#pragma unroll
            for (int e = 0; e < C::HPE; ++e) pr[e] = 0.f;
            const int e_base = hh * C::HPE * C::R;  // first private column of this thread
#pragma unroll
            for (int c = 0; c < C::HPE * C::R / 16; ++c) {
                uint32_t v[16];
                tmem_ld16(tl + a * C::ACC + e_base + 16 * c, v);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int e0 = e_base + 16 * c + 8 * half;  // 8 columns, one 16-byte chunk
                    const int kb = e0 / C::RBLK, x = (e0 % C::RBLK) / 8;
                    const uint4 r4 = *reinterpret_cast<const uint4 *>(
                        rk + kb * (C::TM * C::SWZ) + ((x ^ sw) << 4));
                    const int hx = (16 * c + 8 * half) / C::R;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t rw = u4_word(r4, q);
                        pr[hx] = fmaf(__uint_as_float(v[8 * half + 2 * q]), bf16lo(rw), pr[hx]);
                        pr[hx] = fmaf(__uint_as_float(v[8 * half + 2 * q + 1]), bf16hi(rw), pr[hx]);
                    }
                }
            }
            uint32_t sv[8];
            tmem_ld8(tl + a * C::ACC + C::SH_COL, sv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[a]);
                mbar_arrive(&rkfree[rb]);
            }
            if (q.g >= 0) {
                float o[C::HPE];
#pragma unroll
                for (int e = 0; e < C::HPE; ++e)
                    o[e] = __uint_as_float(sv[hh * C::HPE + e]) +
                           __uint_as_float(sv[C::HPC + hh * C::HPE + e]) + q.winv[e] * pr[e];
                float *dst = P.sc_out + q.g * C::H + h0;
                if constexpr (C::HPE == 2)
                    *reinterpret_cast<float2 *>(dst) = make_float2(o[0], o[1]);
                else
                    dst[0] = o[0];
            }
            return true;
        };
        while (!w.done && ok) {
            if (w.seg != seg_cur) {
                seg_cur = w.seg;
#pragma unroll
                for (int e = 0; e < C::HPE; ++e) winv[e] = __ldg(P.wsc + (size_t)w.b * C::H + h0 + e);
            }
            // turn the tile's two S_K halves in place
            for (int kh = 0; kh < 2; ++kh) {
                const int k = it + kh, s = k % C::STAGES;
                if (!mbar_wait(&full[s], (k / C::STAGES) & 1)) {
                    if (lane == 0) status_or(P.status, LRKV_STATUS_TIMEOUT);
                    ok = false;
                    break;
                }
                uint8_t *st = smem + s * C::STAGE;
                const uint4 *cs = reinterpret_cast<const uint4 *>(st);
                uint4 *sk = reinterpret_cast<uint4 *>(st + C::HALF);
#pragma unroll 4
                for (int c = ew * 32 + lane; c < C::HALF / 16; c += C::EPI * 32) {
                    const uint4 x = sk[c], y = cs[c];
                    sk[c] = make_uint4(turn_pair(x.x, y.x), turn_pair(x.y, y.y), turn_pair(x.z, y.z),
                                       turn_pair(x.w, y.w));
                }
                fence_proxy_async_smem();  // the products read these bytes next
                __syncwarp();
                if (lane == 0) mbar_arrive(&turned[s]);
            }
            if (!ok) break;
            // finish the previous tile while this one's products run
            if (pd.on && !finish(pd)) {
                ok = false;
                break;
            }
            const int j = w.t + row;
            pd.on = true;
            pd.i = i;
            pd.g = (j >= w.t_a && j < w.t_b) ? (int64_t)w.base + j : -1;
#pragma unroll
            for (int e = 0; e < C::HPE; ++e) pd.winv[e] = winv[e];
            it += 2;
            ++i;
            walk_next(w, rg, C::TM);
        }
        if (pd.on && ok) finish(pd);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
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

// Encoded tensor maps depend only on (address, shape, type, box): a small
// per-thread cache of recent encodings saves the host the encode calls of
// every decode.
struct MapKey {
    const void *p;
    int64_t rows;
    int cols, eb, box, kind;
    bool operator==(const MapKey &o) const {
        return p == o.p && rows == o.rows && cols == o.cols && eb == o.eb && box == o.box &&
               kind == o.kind;
    }
};

template <class Encode>
static bool encode_cached(CUtensorMap *map, const MapKey &key, Encode &&encode) {
    constexpr int N = 16;
    struct Entry {
        MapKey key;
        CUtensorMap map;
        bool ok;
    };
    thread_local Entry cache[N] = {};
    thread_local int next = 0;
    for (const Entry &e : cache)
        if (e.ok && e.key == key) {
            *map = e.map;
            return true;
        }
    if (!encode(map)) return false;
    cache[next].key = key;
    cache[next].map = *map;
    cache[next].ok = true;
    next = (next + 1) % N;
    return true;
}

// Map over a pool viewed as [rows, cols] elements of eb bytes (bf16, f16 or
// 8-bit codes), as three dimensions (128 / eb columns, rows, cols * eb / 128
// blocks of 128 bytes) with strides (eb, cols * eb, 128 bytes).  A box of
// (128 / eb) x 16 x box_blocks (default: all blocks) with 128-byte swizzle
// lands a 16-row tile as consecutive 16-row x 128-byte boxes (matches
// box_chunk).
static bool make_map(CUtensorMap *map, const void *pool, int64_t rows, int cols, int eb,
                     int box_blocks = 0, bool f16 = false, int box_rows = 16) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    const int per = 128 / eb, blocks = cols * eb / 128;
    const int bb = box_blocks ? box_blocks : blocks;
    return encode_cached(map, MapKey{pool, rows, cols, eb, bb * 1024 + box_rows, f16 ? 1 : 0}, [&](CUtensorMap *m) {
        cuuint64_t dims[3] = {(cuuint64_t)per, (cuuint64_t)rows, (cuuint64_t)blocks};
        cuuint64_t strides[2] = {(cuuint64_t)cols * eb, 128};
        cuuint32_t box[3] = {(cuuint32_t)per, (cuuint32_t)box_rows, (cuuint32_t)bb};
        cuuint32_t estr[3] = {1, 1, 1};
        const CUtensorMapDataType dt = eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                       : f16   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        return enc(m, dt, 3, const_cast<void *>(pool), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    });
}

// Map over a bf16 pool [rows, cols] as (blk, rows, cols / blk) with blocks
// of blk = 64 (128-byte swizzle) or 32 (64-byte swizzle) elements; a box of
// blk x box_rows x 1 lands one block of box_rows rows.
static bool make_block_map(CUtensorMap *map, const void *pool, int64_t rows, int cols, int blk,
                           int box_rows) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    return encode_cached(map, MapKey{pool, rows, cols, 2, blk * 1024 + box_rows, 3}, [&](CUtensorMap *m) {
        cuuint64_t dims[3] = {(cuuint64_t)blk, (cuuint64_t)rows, (cuuint64_t)(cols / blk)};
        cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)blk * 2};
        cuuint32_t box[3] = {(cuuint32_t)blk, (cuuint32_t)box_rows, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   blk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    });
}

// Map over a row-major [rows, H] array of elements of eb bytes (bf16 joint
// key norms, fp32 given scores) as (H, rows, 1): a box of H x 16 x 1 lands a
// tile's 16 rows, unswizzled.
static bool make_row_map(CUtensorMap *map, const void *base, int64_t rows, int H, int eb,
                         int box_rows = 16) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    return encode_cached(map, MapKey{base, rows, H, eb, box_rows, 2}, [&](CUtensorMap *m) {
        cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)rows, 1};
        cuuint64_t strides[2] = {(cuuint64_t)H * eb, (cuuint64_t)H * eb * rows};
        cuuint32_t box[3] = {(cuuint32_t)H, (cuuint32_t)box_rows, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        const CUtensorMapDataType dt = eb == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    });
}

template <int H, int R, bool Q8 = false, bool GS = false, int NGRP = 1>
struct Pick {
    static constexpr int stage = FastCfg<H, R, 1, Q8, GS, NGRP>::STAGE;
    static constexpr int misc = FastCfg<H, R, 1, Q8, GS, NGRP>::SMEM - FastCfg<H, R, 1, Q8, GS, NGRP>::OFF_BAR;
    static constexpr int fit = (227 * 1024 - misc) / stage;
    // deeper rings of large stages measured slower (more DRAM queueing for
    // the same consumption rate): 3 stages of >= 48 KB, else up to 4; the
    // smaller stages of an 8-bit cache or of given scores keep about as many
    // bytes in flight
    static constexpr int cap = (Q8 || GS) ? (stage >= 24 * 1024 ? 6 : 8) : (stage >= 48 * 1024 ? 3 : 4);
    static constexpr int STAGES = fit > cap ? cap : fit;
    using Cfg = FastCfg<H, R, STAGES, Q8, GS, NGRP>;
};

// Parameters every kernel of the tensor-core decode reads.
static FastParams fast_params(const DecodeArgs &a, const DecodeWs &ws) {
    const auto &c = a.cache;
    FastParams P;
    P.q = static_cast<const __nv_bfloat16 *>(a.q);
    P.seq_lens = a.seq_lens;
    P.page_table = a.page_table;
    P.req_row = a.req_row;
    P.max_pages = a.max_pages;
    P.num_pages = c.num_pages;
    P.page_size = c.page_size;
    P.B = a.B;
    P.scale_log2 = 1.4426950408889634f / sqrtf(128.f);
    P.ws = ws;
    P.status = a.status;
    P.sc = c.dtype == LRKV_FP8_E4M3 ? make_float4(c.scale[0], c.scale[1], c.scale[2], c.scale[3])
                                    : make_float4(1.f, 1.f, 1.f, 1.f);
    P.norm = c.N_K != nullptr;
    P.max_len = decode_max_len(a);
    P.wt = a.rope_ws.wt;
    P.qb = a.rope_ws.qb;
    P.wsc = a.rope_ws.wsc;
    P.sc_out = a.rope_ws.sc;
    P.step_rows = a.early;
    P.B_K = static_cast<const __nv_bfloat16 *>(a.B_K);
    P.B_V = static_cast<const __nv_bfloat16 *>(a.B_V);
    P.out = static_cast<__nv_bfloat16 *>(a.out);
    return P;
}

template <int H, int R, bool Q8, bool GS = false, int NGRP = 1>
static cudaError_t launch_fast_cfg(const DecodeArgs &a, const DecodeWs &ws, int G) {
    using C = typename Pick<H, R, Q8, GS, NGRP>::Cfg;
    static_assert(Pick<H, R, Q8, GS, NGRP>::STAGES >= 2, "at least double buffering");
    const auto &c = a.cache;
    FastMaps maps;
    const int64_t rows = (int64_t)c.num_pages * c.page_size;
    if (!make_map(&maps.sv, c.S_V, rows, 128 * NGRP, C::EB, 0, false, C::TS) ||
        !make_map(&maps.rv, c.R_V, rows, H * R, C::EB, 0, false, C::TS))
        return cudaErrorInvalidValue;
    if (GS) {
        if (!make_row_map(&maps.nk, a.rope_ws.sc, a.rope_ws.sc_rows, H, 4, C::TS)) return cudaErrorInvalidValue;
    } else if (!make_map(&maps.sk, c.S_K, rows, 128 * NGRP, C::EB, 0, false, C::TS) ||
               !make_map(&maps.rk, c.R_K, rows, H * R, C::EB, 0, false, C::TS)) {
        return cudaErrorInvalidValue;
    }
    if (!GS && c.N_K && !make_row_map(&maps.nk, c.N_K, rows, H, 2, C::TS)) return cudaErrorInvalidValue;
    auto kern = decode_split_fast_kernel<C>;
    cudaError_t e = smem_limit_once(kern, C::SMEM);
    if (e != cudaSuccess) return e;
    FastParams P = fast_params(a, ws);
    if (GS) P.norm = 0;
    return launch_pdl(kern, dim3(G), dim3(C::NT), C::SMEM, a.stream, maps, P);
}

#define LRKV_FAST_SHAPES(X) X(16, 16) X(16, 32) X(16, 48) X(16, 56) X(16, 64) X(32, 16) X(32, 32)

// Shapes the tensor-core decode serves with two shared groups (bf16).
#define LRKV_FAST_SHAPES_G2(X) X(16, 32) X(16, 48)

bool fast_decode_supported(int H, int d_h, int r, int page_size, int dtype, int groups) {
    if (groups == 2) {
        if (dtype != LRKV_BF16 || d_h != 128 || page_size % 16 != 0 || !get_encode_tiled()) return false;
#define X(h, rr) if (H == h && r == rr) return true;
        LRKV_FAST_SHAPES_G2(X)
#undef X
        return false;
    }
    if (groups != 1) return false;
    // a tile (16 rows, 32 for 8-bit codes) stays inside a page
    if ((dtype != LRKV_BF16 && dtype != LRKV_FP8_E4M3) || d_h != 128 ||
        page_size % (dtype == LRKV_FP8_E4M3 ? 32 : 16) != 0)
        return false;
    if (!get_encode_tiled()) return false;
#define X(h, rr) if (H == h && r == rr) return true;
    LRKV_FAST_SHAPES(X)
#undef X
    return false;
}

int fast_decode_grid(int, int) { return device_sm_count(); }

cudaError_t launch_split_fast(const DecodeArgs &a, const DecodeWs &ws, int G) {
    const int H = a.cache.H, r = a.cache.r;
    const bool q8 = a.cache.dtype == LRKV_FP8_E4M3, gs = a.rope_ws.wt != nullptr;
    if (cache_groups(a.cache) == 2) {
#define X(h, rr) \
        if (H == h && r == rr) return launch_fast_cfg<h, rr, false, false, 2>(a, ws, G);
        LRKV_FAST_SHAPES_G2(X)
#undef X
        return cudaErrorInvalidValue;
    }
#define X(h, rr)                                                                  \
    if (H == h && r == rr)                                                        \
        return gs ? launch_fast_cfg<h, rr, false, true>(a, ws, G)                 \
             : q8 ? launch_fast_cfg<h, rr, true>(a, ws, G)                        \
                  : launch_fast_cfg<h, rr, false>(a, ws, G);
    LRKV_FAST_SHAPES(X)
#undef X
    return cudaErrorInvalidValue;
}

// ---- exact RoPE: rotary score kernel, then the given-score split kernel

bool rope_fast_supported(int H, int d_h, int r, int page_size, int dtype) {
    // the score kernel lands its 128-row tiles in pieces of 32 or more rows,
    // each inside one page
    return dtype == LRKV_BF16 && r >= 8 && H % rope_tc_heads_per_cta(r) == 0 &&
           page_size % 32 == 0 && fast_decode_supported(H, d_h, r, page_size, dtype);
}

template <int H, int R>
static cudaError_t launch_rope_cfg(const DecodeArgs &a, const DecodeWs &ws) {
    using C = RtcCfg<H, R>;
    const auto &c = a.cache;
    const int64_t rows = (int64_t)c.num_pages * c.page_size;
    // S_K lands in pieces of br rows, each inside a page
    const int br = c.page_size % 128 == 0 ? 128 : c.page_size % 64 == 0 ? 64 : 32;
    RtcMaps m;
    if (!make_map(&m.tab, a.rope16, a.rope_max_pos, 128, 2, 1, true, C::TM) ||
        !make_map(&m.sk, c.S_K, rows, 128, 2, 1, false, br) ||
        !make_block_map(&m.rk, c.R_K, rows, H * R, C::RBLK, br) ||
        !make_map(&m.wt, a.rope_ws.wt, (int64_t)a.B * H * R, 128, 2, 0, true, C::NPRIV) ||
        !make_map(&m.qb, a.rope_ws.qb, (int64_t)a.B * C::NG * 16, 128, 2, 0, false, 16))
        return cudaErrorInvalidValue;
    auto kern = rope_scores_tc_kernel<C>;
    cudaError_t e = smem_limit_once(kern, C::SMEM);
    if (e != cudaSuccess) return e;
    const FastParams P = fast_params(a, ws);
    const int ranges = std::max(1, device_sm_count() / C::NG);
    return launch_pdl(kern, dim3(ranges * C::NG), dim3(C::NT), C::SMEM, a.stream, m, P, br);
}

cudaError_t launch_rope_scores(const DecodeArgs &a, const DecodeWs &ws) {
    const int H = a.cache.H, r = a.cache.r;
#define X(h, rr) \
    if (H == h && r == rr) return launch_rope_cfg<h, rr>(a, ws);
    LRKV_FAST_SHAPES(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace lrkv
