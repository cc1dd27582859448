// lmkv_fp8.cuh -- sm_103a kernels of the fp8-e4m3 quantising gather and
// dequantising scatter.
//
// The quantising gather fuses a cast to float8_e4m3fn, one byte per element
// ("LMCache 分布式 KV Cache 序列化框架：Serde 双层接口设计与自定义扩展实战", section
// 7.1), into the gather of lmkv_kernels.cuh, with one fp32 scale amax / 448
// per (chunk, K/V, layer) tile.  A tile's codes need the whole tile's absmax,
// so each tile is held on chip (registers and shared memory) by a cluster of
// CTAs, whose maxima are exchanged through distributed shared memory: HBM is
// read once.  The dequantising scatter is a copy kernel that widens the codes.
#pragma once

#include "lmkv_kernels.cuh"

#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <cooperative_groups.h>
#include <type_traits>

namespace lmkv {

// ---------------------------------------------------------------------------
// TMA bulk-copy and mbarrier primitives (inline PTX).
__device__ __forceinline__ uint32_t smem_addr(const void* ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase: false if it did not complete within
// `limit_ns` of the global timer (and at most 2^30 polls, should the timer
// not advance).  A bulk copy of at most a few hundred KiB lands in
// microseconds; the first limit (kWaitNs) is far beyond that, so expiry
// means the copies are not being served at all.
constexpr uint64_t kWaitNs = 1000000000ull;          // 1 s
constexpr uint64_t kDrainWaitNs = 10000000000ull;    // 10 s: copies still in flight after a timeout
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < (1u << 24); ++i) {
#pragma unroll 1
        for (int k = 0; k < 64; ++k)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

__device__ __forceinline__ void bulk_g2s(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(sdst)), "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// fp8 e4m3 quantising gather.  One thread-block cluster of kCluster CTAs per
// tile (chunk g, kv, layer l); CTA `rank` owns rows [rank*R, rank*R + R) of the
// tile (R = ceil(n_g / kCluster)).  Values stay in registers between the
// absmax pass and the quantising pass when the slice fits in
// kThreads * kVPT vectors of 16 bytes; otherwise the rest is re-read.
// The absmax is exchanged through distributed shared memory with one split
// cluster barrier; there is no CTA-wide barrier.
constexpr int kQuantMaxRows = 256;   // rows per CTA slice (chunk_size <= kCluster * 256)

// Running max of |x| over 8 bf16 values, as bf16x2 bit patterns (the sign bit
// cleared, so max.bf16x2 of the magnitudes is exact).  kNanProp: a NaN input
// makes the running value NaN (max.NaN.bf16x2), which the caller detects as a
// bit pattern above +inf (0x7F80); otherwise NaNs are ignored, as the
// definition's amax over the tile's values does.
template <bool kNanProp = true>
__device__ __forceinline__ uint32_t absmax_bf16x8(uint32_t acc, const uint4& v) {
    const uint32_t m = 0x7FFF7FFFu;
    auto as_bf2 = [](uint32_t w) { return *reinterpret_cast<const __nv_bfloat162*>(&w); };
    auto mx = [](__nv_bfloat162 x, __nv_bfloat162 y) { return kNanProp ? __hmax2_nan(x, y) : __hmax2(x, y); };
    __nv_bfloat162 a = mx(as_bf2(v.x & m), as_bf2(v.y & m));
    __nv_bfloat162 b = mx(as_bf2(v.z & m), as_bf2(v.w & m));
    a = mx(mx(a, b), as_bf2(acc));
    return *reinterpret_cast<const uint32_t*>(&a);
}

// Larger of the two halves of a running absmax (bf16 magnitude bit patterns
// order like the values; a NaN half sorts above +inf).
__device__ __forceinline__ uint32_t absmax_halves(uint32_t acc) { return max(acc & 0xFFFFu, acc >> 16); }
constexpr uint32_t kBf16InfBits = 0x7F80u;


// Correctly rounded x / s for a per-tile constant s, from the correctly
// rounded reciprocal r = RN(1/s): q0 = RN(x*r) is within an ulp of x/s, the
// remainder q0*s - x is exact in one FMA, and one correction step
// RN(q0 - rem*r) yields RN(x/s) (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990).  The remainder is exact only while it stays out of the fp32
// subnormal range: it is a multiple of ulp(q0) * ulp(s), which needs
// exponent(q0) + exponent(s) >= -103.  With s >= 2^-90 that holds for every
// |q| >= 2^-13, and quotients below 2^-11 round to a signed e4m3 zero however
// their last bits come out; smaller scales take the IEEE division instead
// (kFastDivMinScale).
//
// The kernel evaluates the steps on y = -x, whose remainder q0*s - y is
// q0*s + x, so the unpacked x is used as it is, and under round-to-nearest
// every zero quotient keeps the sign of y.  e4m3 is sign-magnitude and its
// rounding and saturation are symmetric, so the codes of x / s are those of
// y / s with the sign bit flipped.  Two lanes at a time use the packed fp32
// pipe (mul/fma .f32x2).  The tests compare the codes exhaustively with IEEE
// division over every bf16 input and every scale a bf16 absmax can produce.
// The steps hold for finite x and finite s only: a tile holding a NaN, or an
// infinity (whose scale is then infinite), takes the IEEE division.
constexpr float kFastDivMinScale = 0x1p-90f;

// Whether a tile's codes may take the reciprocal-plus-correction division.
__device__ __forceinline__ bool fast_div_ok(float scale, bool tile_has_nan) {
    return !tile_has_nan && scale >= kFastDivMinScale && scale <= 3.4028234663852886e38f;
}

// Every NaN code of four e4m3 codes (either sign: low seven bits all ones)
// made the canonical 0x7F, as the definition's conversion writes it.
__device__ __forceinline__ uint32_t e4m3x4_canonical_nan(uint32_t c) {
    const uint32_t nan_sign = ((c & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
    return c & ~nan_sign;
}

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Four fp32 values -> four e4m3 codes (round to nearest even, saturating),
// byte i of the result from value i.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r) : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
    return r;
}
__device__ __forceinline__ uint32_t e4m3x4(uint64_t a, uint64_t b) {
    float a0, a1, b0, b1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(b0), "=f"(b1) : "l"(b));
    return e4m3x4(a0, a1, b0, b1);
}

// Per-tile constants of the quantiser.
struct QuantK {
    float scale;
    uint64_t s2;     // {s, s}
    uint64_t nr2;    // {-RN(1/s), -RN(1/s)}
};

__device__ __forceinline__ QuantK make_quant(float scale, bool fast) {
    QuantK k;
    k.scale = scale;
    const float nr = fast ? -__frcp_rn(scale) : 0.0f;
    k.s2 = f2_pack(scale, scale);
    k.nr2 = f2_pack(nr, nr);
    return k;
}

// 8 bf16 values (one 16-byte vector) -> 8 e4m3 codes.
template <bool kFastDiv>
__device__ __forceinline__ uint2 quant_bf16x8(const uint4& v, const QuantK& k) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (kFastDiv) {
            uint64_t q[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint32_t word = w[2 * h + i];
                const uint64_t x2 = f2_pack(__uint_as_float(word << 16),
                                            __uint_as_float(word & 0xFFFF0000u));
                const uint64_t q0 = f2_mul(x2, k.nr2);           // RN(y * r), y = -x
                const uint64_t rem = f2_fma(q0, k.s2, x2);       // q0 * s - y, exact
                q[i] = f2_fma(rem, k.nr2, q0);                   // RN(y / s)
            }
            out[h] = e4m3x4(q[0], q[1]) ^ 0x80808080u;           // codes of x / s
        } else {
            const uint32_t w0 = w[2 * h], w1 = w[2 * h + 1];
            out[h] = e4m3x4_canonical_nan(e4m3x4(__fdiv_rn(__uint_as_float(w0 << 16), k.scale),
                                                 __fdiv_rn(__uint_as_float(w0 & 0xFFFF0000u), k.scale),
                                                 __fdiv_rn(__uint_as_float(w1 << 16), k.scale),
                                                 __fdiv_rn(__uint_as_float(w1 & 0xFFFF0000u), k.scale)));
        }
    }
    return make_uint2(out[0], out[1]);
}

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Where the CTA's vectors come from: vector v of the slice is row v / vpr,
// 16-byte column v % vpr.  With kThreads a multiple of vpr each thread keeps
// one column and steps rows by kThreads / vpr.
struct SliceMap {
    const uint8_t* kv_base;     // pool layer l, K or V half
    const int32_t* bt;          // block-table entries of the chunk (column tok0 / B)
    uint32_t r0, vpr, row_bytes, block_size, num_blocks;
    UDiv bdiv, vdiv;
    __device__ __forceinline__ SliceMap(const uint8_t* kvb, const int32_t* btc, uint32_t r0_,
                                        uint32_t vpr_, uint32_t rb, uint32_t bs, uint32_t nb)
        : kv_base(kvb), bt(btc), r0(r0_), vpr(vpr_), row_bytes(rb), block_size(bs), num_blocks(nb),
          bdiv(bs), vdiv(vpr_) {}
    // Source of slice vector v (row-major over the slice), or null for a bad block.
    __device__ __forceinline__ const uint8_t* src(uint32_t row_local, uint32_t col) const {
        const uint32_t row = r0 + row_local;
        const uint32_t jb = bdiv.div(row);
        const int32_t blk = bt[jb];
        if ((uint32_t)blk >= num_blocks) return nullptr;
        const uint32_t slot = row - jb * block_size;
        return kv_base + ((int64_t)blk * block_size + slot) * row_bytes + col * 16u;
    }
};

// The register-staged quantiser's absmax over its slice (registers, then the
// part re-read from the pool), NaN-propagating or not.
template <bool kNanProp, int kThreads, int kVPT>
__device__ __forceinline__ uint32_t absmax_slice(const uint4 (&regs)[kVPT], uint32_t nvec, const SliceMap& sm,
                                                 bool ptr_ok, bool& bad) {
    uint32_t acc = 0;
#pragma unroll
    for (int u = 0; u < kVPT; ++u) acc = absmax_bf16x8<kNanProp>(acc, regs[u]);
    for (uint32_t v = threadIdx.x + kVPT * kThreads; ptr_ok && v < nvec; v += kThreads) {
        const uint32_t row = sm.vdiv.div(v);
        const uint8_t* src = sm.src(row, v - row * sm.vpr);
        if (src == nullptr) { bad = true; continue; }
        const int4 x = ld_stream(reinterpret_cast<const int4*>(src));
        acc = absmax_bf16x8<kNanProp>(acc, make_uint4((uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w));
    }
    return absmax_halves(acc);
}

// Quantise the CTA's slice from registers (and re-read the part that did not
// fit), writing 8 codes per 16-byte source vector.
template <bool kFastDiv, int kThreads, int kVPT>
__device__ __forceinline__ void quant_slice(const uint4 (&regs)[kVPT], uint32_t valid, uint32_t nvec,
                                            const SliceMap& sm, uint8_t* tile_codes, const QuantK& k) {
#pragma unroll
    for (int u = 0; u < kVPT; ++u) {
        const uint32_t v = threadIdx.x + u * kThreads;
        if (v < nvec && (valid >> u) & 1u) {
            const uint2 q = k.scale == 0.0f ? make_uint2(0, 0) : quant_bf16x8<kFastDiv>(regs[u], k);
            *reinterpret_cast<uint2*>(tile_codes + (int64_t)v * 8) = q;
        }
    }
    for (uint32_t v = threadIdx.x + kVPT * kThreads; v < nvec; v += kThreads) {
        const uint32_t row = sm.vdiv.div(v);
        const uint8_t* src = sm.src(row, v - row * sm.vpr);
        if (src == nullptr) continue;
        const int4 x = ld_stream(reinterpret_cast<const int4*>(src));
        const uint4 xv = make_uint4((uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w);
        const uint2 q = k.scale == 0.0f ? make_uint2(0, 0) : quant_bf16x8<kFastDiv>(xv, k);
        *reinterpret_cast<uint2*>(tile_codes + (int64_t)v * 8) = q;
    }
}

template <class B, int kThreads, int kVPT, int kCluster>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
quant_gather_kernel(const __grid_constant__ B p) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ uint32_t warp_max[2][kThreads / 32];     // [exchange round][warp]
    static_assert(kThreads / 32 <= 32, "one lane per warp slot");
    pdl_launch_dependents();
    pdl_wait();

    const int rank = (int)cluster.block_rank();
    const uint32_t tile = blockIdx.x / kCluster;
    const uint32_t ll = tile % (uint32_t)p.layer_n;
    const uint32_t kv = (tile / (uint32_t)p.layer_n) & 1u;
    const int gl = (int)(tile / (uint32_t)p.layer_n / 2u);
    const int l = p.layer_lo + (int)ll;
    const ChunkRef c = resolve_chunk(p, gl);
    const uint32_t rows_per = (uint32_t)(c.ntok + kCluster - 1) / kCluster;
    const uint32_t r0 = rank * rows_per;
    const uint32_t nrows = (uint32_t)max(0, min(c.ntok, (int)(r0 + rows_per)) - (int)r0);
    const uint32_t vpr = (uint32_t)p.row_bytes >> 4;      // 16-byte vectors per row
    const uint32_t row_elems = (uint32_t)p.row_bytes >> 1;
    const uint32_t nvec = nrows * vpr;
    const int lane = threadIdx.x & 31;

    uint8_t* codes = p.chunk_ptrs[p.chunk_base + gl];
    const uint8_t* lb = p.layer_base[l];
    const bool ptr_ok = codes != nullptr && lb != nullptr &&
                        ((reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(lb)) & 15) == 0;
    if (!ptr_ok && threadIdx.x == 0 && rank == 0) report(p, kStatusBadPointer);
    const SliceMap sm(lb + (int64_t)kv * p.num_blocks * p.block_size * p.row_bytes,
                      p.block_table + (int64_t)c.req_row * p.bt_stride + c.col0,
                      r0, vpr, (uint32_t)p.row_bytes, (uint32_t)p.block_size, (uint32_t)p.num_blocks);

    // Pass 1: load the slice and take the running max of |x| on bf16 bits.
    const bool col_fixed = (kThreads % vpr) == 0;
    const uint32_t t_row = threadIdx.x / vpr, t_col = threadIdx.x - t_row * vpr;
    const uint32_t rstep = kThreads / vpr;
    uint4 regs[kVPT];
    uint32_t valid = 0;
    bool bad = false;
#pragma unroll
    for (int u = 0; u < kVPT; ++u) {
        const uint32_t v = threadIdx.x + u * kThreads;
        regs[u] = make_uint4(0, 0, 0, 0);
        if (ptr_ok && v < nvec) {
            uint32_t row, col;
            if (col_fixed) { row = t_row + u * rstep; col = t_col; }
            else { row = sm.vdiv.div(v); col = v - row * vpr; }
            const uint8_t* src = sm.src(row, col);
            if (src == nullptr) {
                bad = true;
            } else {
                const int4 x = ld_stream(reinterpret_cast<const int4*>(src));
                regs[u] = make_uint4((uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w);
                valid |= 1u << u;
            }
        }
    }
    uint32_t m = absmax_slice<true, kThreads, kVPT>(regs, nvec, sm, ptr_ok, bad);
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) report(p, kStatusBadBlock);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) warp_max[0][threadIdx.x >> 5] = m;

    // Exchange: every warp reads all warp maxima of all CTAs of the cluster.
    constexpr int kSlots = kCluster * (kThreads / 32);
    auto exchange = [&](int round) {
        cluster_arrive_release();
        cluster_wait_acquire();
        uint32_t x = 0;
        for (int i = lane; i < kSlots; i += 32)
            x = max(x, *cluster.map_shared_rank(&warp_max[round][i % (kThreads / 32)],
                                                (unsigned)(i / (kThreads / 32))));
        return __reduce_max_sync(0xFFFFFFFFu, x);
    };
    uint32_t w = exchange(0);
    // A NaN somewhere in the tile (every CTA of the cluster sees the same w):
    // the scale is the absmax over the tile's other values, taken in a second
    // round with NaNs ignored, and the tile takes the IEEE division.
    const bool nan_tile = w > kBf16InfBits;
    if (nan_tile) {
        bool bad2 = false;
        m = __reduce_max_sync(0xFFFFFFFFu, absmax_slice<false, kThreads, kVPT>(regs, nvec, sm, ptr_ok, bad2));
        if (lane == 0) warp_max[1][threadIdx.x >> 5] = m;
        w = exchange(1);
    }
    cluster_arrive_relaxed();          // this CTA's shared memory may be released after everyone arrives

    const float amax = __uint_as_float(w << 16);
    const float scale = __fdiv_rn(amax, 448.0f);
    if (rank == 0 && threadIdx.x == 0 && p.scales != nullptr)
        p.scales[((int64_t)(p.chunk_base + gl) * 2 + kv) * p.num_layers + l] = scale;
    if (ptr_ok) {
        uint8_t* tile_codes = codes + (((int64_t)kv * p.num_layers + l) * c.ntok + r0) * row_elems;
        if (fast_div_ok(scale, nan_tile)) {       // reciprocal + correction
            quant_slice<true, kThreads, kVPT>(regs, valid, nvec, sm, tile_codes, make_quant(scale, true));
        } else {                                  // zero, tiny or infinite scale, or NaNs: IEEE division
            quant_slice<false, kThreads, kVPT>(regs, valid, nvec, sm, tile_codes, make_quant(scale, false));
        }
    }
    cluster_wait_acquire();
}

// Shared-memory passes of the staged quantisers: absmax, then quantisation,
// over a CTA's rows staged contiguously in shared memory.  Rows whose block id
// is out of range were not copied; with kCheckRows they are skipped.
template <bool kFastDiv, bool kCheckRows, int kThreads>
__device__ __forceinline__ void quant_smem_slice(const uint8_t* slice, uint32_t nvec, const UDiv& vdiv,
                                                 const uint32_t* row_ok, uint8_t* tile_codes,
                                                 const QuantK& k) {
    // Two adjacent vectors per step (rows hold an even number of vectors when
    // row bytes are a multiple of 32), so codes go out as 16-byte stores.
    if (!kCheckRows && (nvec & 1u) == 0 && (vdiv.d & 1u) == 0) {
        for (uint32_t v2 = threadIdx.x; v2 < (nvec >> 1); v2 += kThreads) {
            const uint4 a = *reinterpret_cast<const uint4*>(slice + (size_t)v2 * 32);
            const uint4 b = *reinterpret_cast<const uint4*>(slice + (size_t)v2 * 32 + 16);
            const uint2 qa = quant_bf16x8<kFastDiv>(a, k);
            const uint2 qb = quant_bf16x8<kFastDiv>(b, k);
            *reinterpret_cast<uint4*>(tile_codes + (int64_t)v2 * 16) = make_uint4(qa.x, qa.y, qb.x, qb.y);
        }
        return;
    }
    for (uint32_t v = threadIdx.x; v < nvec; v += kThreads) {
        if (kCheckRows) {
            const uint32_t row = vdiv.div(v);
            if (!((row_ok[row >> 5] >> (row & 31)) & 1u)) continue;
        }
        const uint4 x = *reinterpret_cast<const uint4*>(slice + (size_t)v * 16);
        *reinterpret_cast<uint2*>(tile_codes + (int64_t)v * 8) = quant_bf16x8<kFastDiv>(x, k);
    }
}

template <bool kCheckRows, int kThreads, bool kNanProp = true>
__device__ __forceinline__ uint32_t absmax_smem_slice(const uint8_t* slice, uint32_t nvec,
                                                      const UDiv& vdiv, const uint32_t* row_ok) {
    uint32_t acc = 0;
    for (uint32_t v = threadIdx.x; v < nvec; v += kThreads) {
        if (kCheckRows) {
            const uint32_t row = vdiv.div(v);
            if (!((row_ok[row >> 5] >> (row & 31)) & 1u)) continue;
        }
        acc = absmax_bf16x8<kNanProp>(acc, *reinterpret_cast<const uint4*>(slice + (size_t)v * 16));
    }
    return acc;
}

// Warp 0 of a quantiser CTA, once its own rows have arrived: ask the TMA unit
// to bring into L2 the slice of the same-rank CTA of tile t2 (a CTA that
// starts about half a wave of clusters later), so that DRAM keeps working
// while this CTA reduces, waits for its cluster and quantises.  Same lookups
// and checks as the slice's own staging; bad ids and pointers are skipped
// (the owning CTA reports them).
template <int kCluster, class B>
__device__ __forceinline__ void prefetch_slice(const B& p, uint32_t t2, uint32_t rank, int lane) {
    if (t2 >= gridDim.x / kCluster) return;
    const uint32_t row_bytes = (uint32_t)p.row_bytes;
    const uint32_t bs = (uint32_t)p.block_size;
    const uint32_t P = bs / (uint32_t)p.parts;
    const UDiv pdiv(P), qdiv((uint32_t)p.parts);
    const uint32_t ll = t2 % (uint32_t)p.layer_n;
    const uint32_t kv = (t2 / (uint32_t)p.layer_n) & 1u;
    const int gl = (int)(t2 / (uint32_t)p.layer_n / 2u);
    const ChunkRef c = resolve_chunk(p, gl);
    const uint32_t rows_per = (uint32_t)(c.ntok + kCluster - 1) / kCluster;
    const uint32_t r0 = rank * rows_per;
    const uint32_t nrows = (uint32_t)max(0, min(c.ntok, (int)(r0 + rows_per)) - (int)r0);
    const uint8_t* lb = p.layer_base[p.layer_lo + (int)ll];
    if (nrows == 0 || lb == nullptr || (reinterpret_cast<uintptr_t>(lb) & 15)) return;
    const uint8_t* kv_base = lb + (int64_t)kv * p.num_blocks * p.block_size * row_bytes;
    const int32_t* bt = p.block_table + (int64_t)c.req_row * p.bt_stride + c.col0;
    const uint32_t pi_end = pdiv.div(r0 + nrows - 1) + 1;
    for (uint32_t pi = pdiv.div(r0) + lane; pi < pi_end; pi += 32) {
        const uint32_t a = max(r0, pi * P), e = min(r0 + nrows, (pi + 1) * P);
        const uint32_t jb = qdiv.div(pi);
        const int32_t blk = bt[jb];
        if ((uint32_t)blk < (uint32_t)p.num_blocks)
            bulk_prefetch_l2(kv_base + ((int64_t)blk * bs + (a - jb * bs)) * row_bytes, (e - a) * row_bytes);
    }
}

// Staged quantising gather (the default when the staged rows fit in shared
// memory).  One thread-block cluster of kCluster CTAs per (chunk, K/V, layer)
// tile; CTA r owns rows [r*n/kCluster, (r+1)*n/kCluster).  The first h rows of
// the CTA's slice (as many whole rows as kThreads * kVPT 16-byte vectors hold)
// are loaded into registers with ordinary loads while warp 0 looks up the page
// runs of the remaining rows in parallel and issues one cp.async.bulk copy per
// run of at most 32 KiB (a page, or a piece of a larger page) into shared
// memory, completing one mbarrier; both halves are in flight
// together.  The CTA takes the absmax over registers and shared memory, the
// cluster exchanges CTA maxima through distributed shared memory (one split
// cluster barrier; lane r reads CTA r's maximum), and every CTA quantises its
// rows.  Measured on the 8B batch with clusters of 8: 4 register vectors per
// thread (16 KiB of registers + 48 KiB of shared memory per CTA) beat staging
// everything in shared memory (0.394 vs 0.406 ms) and 8 or 12 register
// vectors; clusters of 4 (16 KiB + 112 KiB per CTA, two CTAs per SM) are
// faster again (0.371 ms): half as many CTAs meet at each cluster barrier.
template <class B, int kThreads, int kVPT, int kCluster>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
quant_gather_hybrid_kernel(const __grid_constant__ B p) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(128) uint8_t slice[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t cta_max[2];                    // [exchange round]
    __shared__ uint32_t row_ok[kQuantMaxRows / 32];
    __shared__ uint32_t any_bad;
    static_assert(kCluster <= 32, "one lane per cluster rank");
    pdl_launch_dependents();
    pdl_wait();

    const uint32_t rank = cluster.block_rank();
    const uint32_t tile = blockIdx.x / kCluster;
    const uint32_t ll = tile % (uint32_t)p.layer_n;
    const uint32_t kv = (tile / (uint32_t)p.layer_n) & 1u;
    const int gl = (int)(tile / (uint32_t)p.layer_n / 2u);
    const int l = p.layer_lo + (int)ll;
    const ChunkRef c = resolve_chunk(p, gl);
    const uint32_t rows_per = (uint32_t)(c.ntok + kCluster - 1) / kCluster;
    const uint32_t r0 = rank * rows_per;
    const uint32_t nrows = (uint32_t)max(0, min(c.ntok, (int)(r0 + rows_per)) - (int)r0);
    const uint32_t row_bytes = (uint32_t)p.row_bytes;
    const uint32_t vpr = row_bytes >> 4;
    const uint32_t h = min(nrows, (uint32_t)(kThreads * kVPT) / vpr);   // rows held in registers
    const uint32_t nvec_reg = h * vpr;
    const uint32_t nrows_s = nrows - h;                                   // rows staged in shared memory
    const uint32_t nvec_s = nrows_s * vpr;
    const int lane = threadIdx.x & 31;

    uint8_t* codes = p.chunk_ptrs[p.chunk_base + gl];
    const uint8_t* lb = p.layer_base[l];
    const bool ptr_ok = codes != nullptr && lb != nullptr &&
                        ((reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(lb)) & 15) == 0;
    const SliceMap sm(lb + (int64_t)kv * p.num_blocks * p.block_size * row_bytes,
                      p.block_table + (int64_t)c.req_row * p.bt_stride + c.col0, r0, vpr, row_bytes,
                      (uint32_t)p.block_size, (uint32_t)p.num_blocks);
    if (threadIdx.x < 32) {
        // Warp 0 stages rows [r0 + h, r0 + nrows) in shared memory.
        if (lane == 0) {
            if (!ptr_ok && rank == 0) report(p, kStatusBadPointer);
            cta_max[0] = cta_max[1] = 0;
            mbar_init(&bar, 1);
            fence_barrier_init();
        }
        for (int i = lane; i < kQuantMaxRows / 32; i += 32) row_ok[i] = 0;
        __syncwarp();
        // One bulk copy per piece of P = block_size / parts rows (pages of at
        // most 32 KiB are one piece; larger pages are cut so that several
        // copies are in flight, as with small pages).  Piece i covers slice
        // rows [i*P, (i+1)*P), inside page i / parts.
        const uint32_t bs = (uint32_t)p.block_size;
        const uint32_t P = bs / (uint32_t)p.parts;
        const UDiv pdiv(P), qdiv((uint32_t)p.parts);
        const uint32_t s0 = r0 + h;
        const uint32_t pi0 = nrows_s ? pdiv.div(s0) : 0u;
        const uint32_t pi_end = nrows_s ? pdiv.div(s0 + nrows_s - 1) + 1 : 0u;
        uint32_t bytes = 0;
        bool bad = false;
        for (uint32_t pi = pi0 + lane; ptr_ok && pi < pi_end; pi += 32) {
            const uint32_t a = max(s0, pi * P), e = min(s0 + nrows_s, (pi + 1) * P);
            const int32_t blk = sm.bt[qdiv.div(pi)];
            if ((uint32_t)blk < (uint32_t)p.num_blocks) {
                bytes += (e - a) * row_bytes;
                for (uint32_t r = a - s0; r < e - s0; ++r) atomicOr(&row_ok[r >> 5], 1u << (r & 31));
            } else {
                bad = true;
            }
        }
        const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, bytes);
        const bool any = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0) {
            any_bad = any ? 1u : 0u;
            mbar_arrive_expect_tx(&bar, total);
        }
        __syncwarp();
        for (uint32_t pi = pi0 + lane; ptr_ok && pi < pi_end; pi += 32) {
            const uint32_t a = max(s0, pi * P), e = min(s0 + nrows_s, (pi + 1) * P);
            const uint32_t jb = qdiv.div(pi);
            const int32_t blk = sm.bt[jb];
            if ((uint32_t)blk < (uint32_t)p.num_blocks)
                bulk_g2s(slice + (size_t)(a - s0) * row_bytes,
                         sm.kv_base + ((int64_t)blk * bs + (a - jb * bs)) * row_bytes, (e - a) * row_bytes, &bar);
        }
    }
    // Every thread: rows [r0, r0 + h) into registers.
    const bool col_fixed = (kThreads % vpr) == 0;
    const uint32_t t_row = threadIdx.x / vpr, t_col = threadIdx.x - t_row * vpr;
    const uint32_t rstep = kThreads / vpr;
    uint4 regs[kVPT];
    uint32_t valid = 0;
    bool bad_reg = false;
#pragma unroll
    for (int u = 0; u < kVPT; ++u) {
        const uint32_t v = threadIdx.x + u * kThreads;
        regs[u] = make_uint4(0, 0, 0, 0);
        if (ptr_ok && v < nvec_reg) {
            uint32_t row, col;
            if (col_fixed) { row = t_row + u * rstep; col = t_col; }
            else { row = sm.vdiv.div(v); col = v - row * vpr; }
            const uint8_t* src = sm.src(row, col);
            if (src == nullptr) {
                bad_reg = true;
            } else {
                const int4 x = ld_stream(reinterpret_cast<const int4*>(src));
                regs[u] = make_uint4((uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w);
                valid |= 1u << u;
            }
        }
    }
    if (__any_sync(0xFFFFFFFFu, bad_reg) && lane == 0) report(p, kStatusBadBlock);
    __syncthreads();                                  // barrier initialised, row_ok / any_bad written
    // The bulk copies land in microseconds.  Should they not complete within
    // the first bound, the CTA reports LMKV_ERR_TIMEOUT, writes no codes, and
    // keeps waiting (a further, longer bound) so that it does not exit while
    // its copies may still write into its shared memory.
    bool timed_out = false;
    if (!mbar_wait_bounded(&bar, 0)) {
        timed_out = true;
        if (threadIdx.x == 0) report(p, kStatusTimeout);
        (void)mbar_wait_bounded(&bar, 0, kDrainWaitNs);
    }
    if (threadIdx.x == 0 && any_bad) report(p, kStatusBadBlock);
    if (p.prefetch_ahead > 0 && threadIdx.x < 32)
        prefetch_slice<kCluster>(p, tile + (uint32_t)p.prefetch_ahead, rank, lane);
    const bool check_rows = any_bad != 0;
    // CTA maximum of |x| over registers and shared memory, NaN-propagating
    // (kNanProp) or NaN-ignoring, into cta_max[round].
    auto cta_absmax = [&](auto nan_prop, int round) {
        constexpr bool kNP = decltype(nan_prop)::value;
        uint32_t acc = 0;
#pragma unroll
        for (int u = 0; u < kVPT; ++u) acc = absmax_bf16x8<kNP>(acc, regs[u]);
        const uint32_t a2 = check_rows ? absmax_smem_slice<true, kThreads, kNP>(slice, nvec_s, sm.vdiv, row_ok)
                                       : absmax_smem_slice<false, kThreads, kNP>(slice, nvec_s, sm.vdiv, row_ok);
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max(absmax_halves(acc), absmax_halves(a2)));
        if (lane == 0) atomicMax(&cta_max[round], m);
    };
    auto exchange = [&](int round) {
        cluster_arrive_release();
        cluster_wait_acquire();
        const uint32_t x = lane < kCluster ? *cluster.map_shared_rank(&cta_max[round], (unsigned)lane) : 0u;
        return __reduce_max_sync(0xFFFFFFFFu, x);
    };
    cta_absmax(std::true_type{}, 0);
    uint32_t w = exchange(0);
    // A NaN somewhere in the tile (every CTA of the cluster sees the same w):
    // the scale is the absmax over the tile's other values, taken in a second
    // round with NaNs ignored, and the tile takes the IEEE division.
    const bool nan_tile = w > kBf16InfBits;
    if (nan_tile) {
        cta_absmax(std::false_type{}, 1);
        w = exchange(1);
    }
    cluster_arrive_relaxed();          // this CTA's shared memory may be released after everyone arrives

    const float amax = __uint_as_float(w << 16);
    const float scale = __fdiv_rn(amax, 448.0f);
    if (rank == 0 && threadIdx.x == 0 && p.scales != nullptr)
        p.scales[((int64_t)(p.chunk_base + gl) * 2 + kv) * p.num_layers + l] = scale;
    if (ptr_ok && !timed_out) {
        uint8_t* tile_codes = codes + (((int64_t)kv * p.num_layers + l) * c.ntok + r0) * (row_bytes >> 1);
        uint8_t* smem_codes = tile_codes + (size_t)nvec_reg * 8;
        const bool fast = fast_div_ok(scale, nan_tile);
        const QuantK k = make_quant(scale, fast);
        // register rows
#pragma unroll
        for (int u = 0; u < kVPT; ++u) {
            const uint32_t v = threadIdx.x + u * kThreads;
            if (v < nvec_reg && (valid >> u) & 1u) {
                const uint2 q = scale == 0.0f ? make_uint2(0, 0)
                              : fast ? quant_bf16x8<true>(regs[u], k) : quant_bf16x8<false>(regs[u], k);
                *reinterpret_cast<uint2*>(tile_codes + (int64_t)v * 8) = q;
            }
        }
        // shared-memory rows
        if (scale == 0.0f) {
            for (uint32_t v = threadIdx.x; v < nvec_s; v += kThreads) {
                const uint32_t row = sm.vdiv.div(v);
                if (!check_rows || ((row_ok[row >> 5] >> (row & 31)) & 1u))
                    *reinterpret_cast<uint2*>(smem_codes + (int64_t)v * 8) = make_uint2(0, 0);
            }
        } else if (fast) {
            if (check_rows) quant_smem_slice<true, true, kThreads>(slice, nvec_s, sm.vdiv, row_ok, smem_codes, k);
            else quant_smem_slice<true, false, kThreads>(slice, nvec_s, sm.vdiv, row_ok, smem_codes, k);
        } else {
            quant_smem_slice<false, true, kThreads>(slice, nvec_s, sm.vdiv, row_ok, smem_codes, k);
        }
    }
    cluster_wait_acquire();
}

// ---------------------------------------------------------------------------
// fp8 e4m3 dequantising scatter: per item (chunk, kv, layer, block part),
// 8 codes (8 bytes) in, 8 bf16 (16 bytes) out per thread step.
__device__ __forceinline__ uint2 ld_stream8(const uint2* ptr) {
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(ptr));
    return r;
}

__device__ __forceinline__ uint32_t dequant_pair(uint16_t two_codes, float scale) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two_codes, __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    return *reinterpret_cast<const uint32_t*>(&b);
}

template <class B, int kThreads, int kUnroll>
__global__ void __launch_bounds__(kThreads)
dequant_scatter_kernel(const __grid_constant__ B p, int64_t num_items) {
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t item = blockIdx.x; item < num_items; item += gridDim.x) {
        // Decode the item against a bf16 pool, then derive the code run from it.
        Run run;
        if (!item_run(p, item, run)) continue;
        const int kv = run.kv, gl = run.gl;
        const int l = p.layer_lo + run.ll;
        const float scale = p.scales[((int64_t)(p.chunk_base + gl) * 2 + kv) * p.num_layers + l];
        // chunk-side offset of the run in bf16 bytes -> the same rows in code bytes
        const uint8_t* cb = p.chunk_ptrs[p.chunk_base + gl];
        const int64_t code_off = (run.chunk - cb) >> 1;
        // 8 codes (8 bytes) per thread step -> one 16-byte store, so that a
        // warp's store instruction covers 512 contiguous bytes; kUnroll code
        // words per thread are loaded before their stores (the code and pool
        // pointers may alias, so the compiler never moves a load above an
        // earlier store by itself)
        const int n8 = (int)(run.bytes >> 4);
        const uint2* src = reinterpret_cast<const uint2*>(cb + code_off);
        int4* dst = reinterpret_cast<int4*>(run.pool);
        for (int base = threadIdx.x; base < n8; base += kThreads * kUnroll) {
            uint2 ci[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = base + u * kThreads;
                if (v < n8) ci[u] = ld_stream8(src + v);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = base + u * kThreads;
                if (v >= n8) continue;
                st_stream(dst + v, make_int4((int)dequant_pair((uint16_t)(ci[u].x & 0xFFFFu), scale),
                                             (int)dequant_pair((uint16_t)(ci[u].x >> 16), scale),
                                             (int)dequant_pair((uint16_t)(ci[u].y & 0xFFFFu), scale),
                                             (int)dequant_pair((uint16_t)(ci[u].y >> 16), scale)));
            }
        }
    }
}

}  // namespace lmkv
