// Shared device helpers for the LRKV kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lrkv.h"

namespace lrkv {

// ---------------------------------------------------------------------------
// Launch plan shared by the decode kernels.
//
// Decode work is balanced over a fixed grid of G CTAs: the visible rows of
// all requests are laid end to end (request b occupies [off[b], off[b+1])),
// and CTA g takes the contiguous range [g*chunk, (g+1)*chunk).  A CTA's range
// can cut several requests; each (request, CTA) piece is a "segment" whose
// partial softmax state goes to slot b + g (unique among the segments that
// exist, so B + G slots suffice).
// ---------------------------------------------------------------------------
struct DecodePlan {
    int32_t total;   // sum of the (validated) sequence lengths
    int32_t chunk;   // rows per CTA (multiple of the tile size)
    int32_t pad[2];
    // int32_t off[B + 1] follows
};

constexpr int kPlanTileAlign = 16;

// Workspace layout of lrkv_decode (all offsets 256-byte aligned):
//   [plan header + off[B+1] + cnt[4]] [p: B*H*r f32] [ml: slots*H*2 f32]
//   [acc: slots*H*(d_h+r) f32]
// cnt[0] counts the CTAs of the tensor-core split kernel that have written
// all their partial states (the merge phase starts when it reaches the grid
// size); the prologue zeroes it.  cnt[1..3] are spare.
constexpr int kDecodeCounters = 4;

struct DecodeWs {
    DecodePlan *plan;
    int32_t *off;
    int32_t *cnt;
    float *p;
    float *ml;
    float *acc;
    size_t bytes;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Shared key/value groups of a cache (0 and 1 both mean one shared basis);
// head h reads group h / (H / groups).
__host__ __device__ inline int cache_groups(const lrkv_cache_t &c) { return c.G > 1 ? c.G : 1; }

__host__ __device__ inline DecodeWs decode_ws_layout(void *base, int B, int H, int d_h, int r,
                                                     int G) {
    DecodeWs w;
    char *p = static_cast<char *>(base);
    size_t o = 0;
    w.plan = reinterpret_cast<DecodePlan *>(p + o);
    w.off = reinterpret_cast<int32_t *>(p + o + sizeof(DecodePlan));
    w.cnt = w.off + (B + 1);
    o += align256(sizeof(DecodePlan) + sizeof(int32_t) * (size_t)(B + 1 + kDecodeCounters));
    w.p = reinterpret_cast<float *>(p + o);
    o += align256(sizeof(float) * (size_t)B * H * r);
    size_t slots = (size_t)B + G;
    w.ml = reinterpret_cast<float *>(p + o);
    o += align256(sizeof(float) * slots * H * 2);
    w.acc = reinterpret_cast<float *>(p + o);
    o += align256(sizeof(float) * slots * H * (size_t)(d_h + r));
    w.bytes = o;
    return w;
}

// Heads of one CTA of the tensor-core rotary score kernel: its private
// products C_j W_h of those heads form one MMA of N = heads * r columns, at
// most 224 (the rest of a 256-column accumulator holds the shared term).
__host__ __device__ constexpr int rope_tc_heads_per_cta(int r) { return 4 * r <= 224 ? 4 : 2; }

// Extra workspace of the tensor-core rotary decode (lrkv_decode_rope), after
// the decode workspace (all offsets 256-byte aligned):
//   [wt: B*H*r*d_h f16]    per (request, head) the rotated private operand W,
//                          transposed ([r][d_h], d_h contiguous), scaled by a
//                          power of two
//   [qb: B*(H/g)*16*d_h bf16]  per (request, group of g heads) the rotated
//                          queries q D_i as rows: row i the bf16 value of head
//                          i of the group, row g + i the bf16 remainder, rows
//                          2g .. 15 zero (g = rope_tc_heads_per_cta(r))
//   [wsc: B*H f32]         inverse scale of each W
//   [sc: B*max_seq_len*H f32]  raw scores of every visible row, row-major by
//                          the plan's row index (request b's rows start at off[b])
struct RopeFastWs {
    uint16_t *wt;
    uint16_t *qb;
    float *wsc;
    float *sc;
    int64_t sc_rows;
    size_t bytes;
};

__host__ __device__ inline RopeFastWs rope_fast_ws_layout(void *base, int B, int H, int d_h, int r,
                                                          int max_seq_len) {
    RopeFastWs w;
    char *p = static_cast<char *>(base);
    size_t o = 0;
    w.wt = reinterpret_cast<uint16_t *>(p + o);
    o += align256(sizeof(uint16_t) * (size_t)B * H * d_h * r);
    w.qb = reinterpret_cast<uint16_t *>(p + o);
    o += align256(sizeof(uint16_t) * (size_t)B * (H / rope_tc_heads_per_cta(r)) * 16 * d_h);
    w.wsc = reinterpret_cast<float *>(p + o);
    o += align256(sizeof(float) * (size_t)B * H);
    w.sc = reinterpret_cast<float *>(p + o);
    w.sc_rows = (int64_t)B * max_seq_len;
    o += align256(sizeof(float) * (size_t)w.sc_rows * H);
    w.bytes = o;
    return w;
}

// Byte offset of the f16 copy inside a rotary table of max_pos rows: the
// float (cos, sin) pairs come first, [max_pos][d_h/2][2].
__host__ __device__ inline size_t rope_table_f16_offset(int d_h, int max_pos) {
    return align256(sizeof(float) * (size_t)max_pos * d_h);
}

// ---------------------------------------------------------------------------
// Element conversion
// ---------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
    __device__ static float load(const float *p) { return *p; }
    __device__ static void store(float *p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
    __device__ static float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    __device__ static void store(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
};

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// 16-byte vector of T widened to floats (8 bf16 or 4 fp32 elements).
template <typename T> struct Vec16;
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const __nv_bfloat16 *p, float (&v)[8]) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
        v[4] = __uint_as_float(u.z << 16); v[5] = __uint_as_float(u.z & 0xffff0000u);
        v[6] = __uint_as_float(u.w << 16); v[7] = __uint_as_float(u.w & 0xffff0000u);
    }
};
template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ static void load(const float *p, float (&v)[4]) {
        const float4 u = *reinterpret_cast<const float4 *>(p);
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    }
};

// Block-cooperative copy of n elements (n a multiple of Vec16<T>::N, src
// 16-byte aligned) into fp32 shared memory, several vectors in flight per
// thread.
template <typename T>
__device__ __forceinline__ void stage_f32(float *dst, const T *src, int n) {
    constexpr int V = Vec16<T>::N, U = 4;
    const int nv = n / V, step = blockDim.x * U;
    for (int base = threadIdx.x; base < nv; base += step) {
        float v[U][V];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + u * (int)blockDim.x < nv) Vec16<T>::load(src + (size_t)(base + u * blockDim.x) * V, v[u]);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + u * (int)blockDim.x < nv)
#pragma unroll
                for (int e = 0; e < V; ++e) dst[(base + u * blockDim.x) * V + e] = v[u][e];
    }
}

// ---------------------------------------------------------------------------
// 8-bit E4M3 cache codes (LRKV_FP8_E4M3)
// ---------------------------------------------------------------------------
// Two floats -> two codes (round to nearest even, saturating at +-448; NaN
// stays NaN); `lo` lands in bits 0-7.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// Two codes -> two fp16 values (exact: every E4M3 value is an fp16 value); the
// code in bits 0-7 lands in the low half.
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint16_t codes) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
    return r;
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t code) {
    const uint32_t h2 = f16x2_from_e4m3x2(code);
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}

// Two floats -> f16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Byte permute: result byte i = byte sel_i of the 8-byte value {b:a}.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "n"(SEL));
    return r;
}
// 2^e as a float, for -126 <= e <= 127 (exact).
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }
// Shift e with 2^e * m in [2^14, 2^15) (0 for m = 0 or non-finite m): the
// exact power-of-two scaling that puts values of magnitude <= m in f16 range.
__device__ __forceinline__ int f16_range_shift(float m) {
    if (!(m > 0.f) || !isfinite(m)) return 0;
    const int ex = (int)((__float_as_uint(m) >> 23) & 0xff) - 127;
    return max(-125, min(125, 14 - ex));
}

// Value of one stored cache element, before its pool's scale.
template <typename TC> struct CacheLoad;
template <> struct CacheLoad<float> {
    __device__ static float load(const float *p) { return *p; }
};
template <> struct CacheLoad<__nv_bfloat16> {
    __device__ static float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
};
template <> struct CacheLoad<uint8_t> {
    __device__ static float load(const uint8_t *p) { return e4m3_to_f32(*p); }
};

__device__ __forceinline__ void status_or(int32_t *st, uint32_t bits) {
    if (st) atomicOr(reinterpret_cast<unsigned int *>(st), bits);
}

// ---------------------------------------------------------------------------
// Shared memory / mbarrier / bulk-copy wrappers (PTX ISA, sm_90+)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase.  Returns false if the phase did not
// complete within ~2 s of wall time (the caller then records
// LRKV_STATUS_TIMEOUT and leaves its loop instead of spinning forever).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    uint32_t ok = 0;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((it & 255u) == 255u && globaltimer_ns() - t0 > 2000000000ull) return false;
    }
}

// Bounded wait that suspends the thread in hardware between polls (PTX
// try_wait with a suspend-time hint of `hint_ns`) instead of re-polling the
// barrier word: waiting warps then leave shared-memory bandwidth to the
// tensor cores.  Same 2 s bound and return value as mbar_wait.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity,
                                                uint32_t hint_ns = 20000) {
    const uint32_t a = smem_u32(bar);
    uint32_t ok = 0;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; "
            "selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(a), "r"(parity), "r"(hint_ns)
            : "memory");
        if (ok) return true;
        // the clock is read only once the phase was found incomplete
        if (it == 0) t0 = globaltimer_ns();
        else if (globaltimer_ns() - t0 > 2000000000ull) return false;
    }
}

// 2-D tiled TMA load: box at (x, y) of the tensor map into shared memory,
// completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled TMA load: box at (x, y, z) of the tensor map.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 cache-eviction policy (see l2_evict_first_policy).
__device__ __forceinline__ void tma_load_3d_hint(void *dst, const CUtensorMap *map, int x, int y,
                                                 int z, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 3-D tiled TMA store of a shared-memory box to (x, y, z) of the tensor map,
// tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, int x, int y, int z,
                                             const void *src) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the bulk stores of this thread have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Policy marking streamed data as first to leave L2, so that small tensors
// reused every step (weights, bases, partials) stay resident.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Policy marking data reused every step (weights) as last to leave L2.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 32-bit global load carrying an L2 cache policy.
__device__ __forceinline__ uint32_t ld_u32_hint(const void *ptr, uint64_t policy) {
    uint32_t v;
    asm volatile("ld.global.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(v) : "l"(ptr), "l"(policy));
    return v;
}

// Plain contiguous bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// The same bulk copy with an L2 cache policy on the source reads.
__device__ __forceinline__ void bulk_load_hint(void *dst, const void *src, uint32_t bytes,
                                               uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// preamble, and wait for the previous kernel's completion and memory.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Scope guard of a kernel that works before its dependency wait and has
// already let its dependents launch: when on, the wait runs as the thread
// leaves the scope, on every return path (the grid then completes only after
// its predecessor has).
struct PdlWaitOnExit {
    bool on;
    __device__ ~PdlWaitOnExit() {
        if (on) pdl_wait();
    }
};

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core fragments (m16n8k16, bf16 in, fp32 accumulate)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile
// written by TMA with CU_TENSOR_MAP_SWIZZLE_128B (rows of 128 bytes; the
// chunk index is XORed with the row index modulo 8).
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device.  The attribute belongs to the device that is current when it is
// set, so it is recorded per (kernel, device, size) and set once for each:
// a process that drives several GPUs gets it on every one of them.
cudaError_t smem_limit_once(const void *kern, int bytes);
template <typename... KArgs>
inline cudaError_t smem_limit_once(void (*kern)(KArgs...), int bytes) {
    return smem_limit_once(reinterpret_cast<const void *>(kern), bytes);
}

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while its predecessor in the stream drains; every kernel of this
// library starts with pdl_wait(), so stream order is kept for its reads.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

}  // namespace lrkv
