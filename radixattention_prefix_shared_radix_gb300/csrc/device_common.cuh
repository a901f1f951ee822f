// Device helpers shared by the attention kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "common.h"

namespace sgldev {

using bf16 = __nv_bfloat16;

constexpr int kTile = 64;     // KV positions per pipeline stage
constexpr int kStages = 3;    // stages in flight
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their writes are visible (a no-op without such a
// dependency), and let the grids that depend on this one be scheduled now
// (they wait in turn before touching memory).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
// fetch the line holding `p` (a valid global address) into L1
__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile("prefetch.global.L1 [%0];\n" ::"l"(p)); }

// An L2 policy that evicts the lines it tags first: for data read exactly
// once, so that it does not push the kernels' code and tables out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
// cp_async16 with an L2 cache policy.
__device__ __forceinline__ void cp_async16_pol(uint32_t dst, const void* src, bool valid, uint64_t pol) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(dst), "l"(src), "r"(n),
                 "l"(pol)
                 : "memory");
}
// 4-byte copy (cached in L1), no zero fill.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void st_shared_s32(uint32_t addr, int32_t v) {
    asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ int32_t ld_shared_s32(uint32_t addr) {
    int32_t v;
    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x in one MUFU operation (results below 2^-126 flush to zero, which the
// softmax weights tolerate: they are summed with weights of at least 1).
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// (y0, y1) = (x0, x1) * s + (c, c): one packed fp32x2 FMA (sm_100+).
__device__ __forceinline__ void ffma2_sc(float& y0, float& y1, float x0, float x1, float s, float c) {
    asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %4};\n mov.b64 c, {%5, %5};\n"
        " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
        : "=f"(y0), "=f"(y1)
        : "f"(x0), "f"(x1), "f"(s), "f"(c));
}
// (a0, a1) += (x0, x1): one packed fp32x2 add.
__device__ __forceinline__ void fadd2_acc(float& a0, float& a1, float x0, float x1) {
    asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n add.f32x2 d, a, b;\n"
        " mov.b64 {%0, %1}, d;\n}"
        : "+f"(a0), "+f"(a1)
        : "f"(x0), "f"(x1));
}
// max(a, b, c) in one instruction (sm_100+).
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
// Four FP8 E4M3 values (one 32-bit word) as two f16x2 words, exactly (every
// E4M3 value is an f16 value).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}
// bf16x2 -> f16x2 (query values: in range and exact for N(0,1)-sized data)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
    const float a = __uint_as_float(x << 16), b = __uint_as_float(x & 0xffff0000u);
    uint32_t y;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(y) : "f"(b), "f"(a));
    return y;
}
// The same, noting in `bad` a value that f16 cannot hold: |x| >= 65536 (the
// largest bf16 below it, 65280, is an f16 value), an infinity or a NaN.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_chk(uint32_t x, uint32_t& bad) {
    bad |= ((x & 0x7fffu) >= 0x4780u) | (((x >> 16) & 0x7fffu) >= 0x4780u);
    return bf16x2_to_f16x2(x);
}
// error word bit 3: a query element outside f16's range met an FP8 pool
constexpr uint32_t kErrQRange = 8u;
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t y;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(y) : "f"(hi), "f"(lo));
    return y;
}

// Byte offset of 16-byte chunk c of row r in a swizzled tile of D-wide rows.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// Shared-memory row layouts of a bf16 [rows x D] tile, as byte offsets of
// 16-byte chunk c of row r.  Swz: rows of D*2 bytes, chunk index XOR (r & 7).
// Pad: rows of D*2 + 16 bytes (whole rows land contiguously, e.g. from one
// bulk copy; the 16-byte pad keeps 8 consecutive rows in distinct banks).
template <int D>
struct Swz {
    static __device__ __forceinline__ uint32_t off(int r, int c) { return swz<D>(r, c); }
};
template <int D>
struct Pad {
    static constexpr int RS = D * 2 + 16;
    static __device__ __forceinline__ uint32_t off(int r, int c) { return static_cast<uint32_t>(r * RS + (c << 4)); }
};

__device__ __forceinline__ float quad_max(float v) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

// Slot of position `pos` in row `row`, or -1 (and the error bit) when the
// table entry is outside the pool.
__device__ __forceinline__ int64_t load_slot(const int32_t* r2t, int64_t ld, int row, int pos, int64_t num_slots,
                                             uint32_t* err) {
    const int32_t s = __ldg(r2t + (int64_t)row * ld + pos);
    if (s < 0 || s >= num_slots) {
        atomicOr(err, 1u);
        return -1;
    }
    return s;
}

// ---------------------------------------------------------------------------
// Online-softmax state of one warp over a 16-row m-tile: O accumulators in
// mma C layout (rows g and g+8 of the tile, g = lane / 4), running max m and
// per-thread partial sum l for both rows.
// ---------------------------------------------------------------------------
template <int D>
struct WarpState {
    float o[D / 8][4];
    float m[2];
    float l[2];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
    }
};

// Process NT 8-column score tiles s[NT][4] (already scaled to log2 units and
// masked): update the running max/sum, rescale O and add P V for the tile's
// 16*(NT/2) KV rows starting at smem row vrow0 of sV.
template <int D, int NT, typename L = Swz<D>>
__device__ __forceinline__ void softmax_pv(WarpState<D>& st, float (&s)[NT][4], const uint8_t* sV, int vrow0,
                                           int lane) {
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
        mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
    }
    mx0 = quad_max(mx0);
    mx1 = quad_max(mx1);
    const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
    const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float a0 = exp2f(st.m[0] - mu0), a1 = exp2f(st.m[1] - mu1);
    st.m[0] = mn0;
    st.m[1] = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        s[n][0] = exp2f(s[n][0] - mu0);
        s[n][1] = exp2f(s[n][1] - mu0);
        s[n][2] = exp2f(s[n][2] - mu1);
        s[n][3] = exp2f(s[n][3] - mu1);
        ps0 += s[n][0] + s[n][1];
        ps1 += s[n][2] + s[n][3];
    }
    st.l[0] = st.l[0] * a0 + ps0;
    st.l[1] = st.l[1] * a1 + ps1;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        st.o[n][0] *= a0;
        st.o[n][1] *= a0;
        st.o[n][2] *= a1;
        st.o[n][3] *= a1;
    }
    const uint32_t vbase = smem_u32(sV);
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) {      // 16 KV rows per k-step
        uint32_t a[4];
        a[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
        a[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
        a[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        a[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
        const int vr = vrow0 + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vbase + L::off(vr, dp * 2 + (lane >> 4)), b0, b1, b2, b3);
            mma16816(st.o[2 * dp], a, b0, b1);
            mma16816(st.o[2 * dp + 1], a, b2, b3);
        }
    }
}

// S[16 x 8*NT] = Q(m-tile, fragments qf) * K^T for the NT/2 16-row groups of
// KV rows starting at smem row krow0 of sK.
template <int D, int NT, typename L = Swz<D>>
__device__ __forceinline__ void qk(float (&s)[NT][4], const uint32_t (&qf)[D / 16][4], const uint8_t* sK, int krow0,
                                   int lane) {
#pragma unroll
    for (int n = 0; n < NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
    const uint32_t kbase = smem_u32(sK);
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
        const int kr = krow0 + np * 16 + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + L::off(kr, ks * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
            mma16816(s[2 * np], qf[ks], b0, b1);
            mma16816(s[2 * np + 1], qf[ks], b2, b3);
        }
    }
}

template <int D, typename L = Swz<D>>
__device__ __forceinline__ void load_qfrag(uint32_t (&qf)[D / 16][4], const uint8_t* sQ, int row0, int lane) {
    const uint32_t qbase = smem_u32(sQ);
    const int r = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
        ldsm_x4(qbase + L::off(r, ks * 2 + (lane >> 4)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
}

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy primitives.  Every wait is bounded: after kSpinLimit
// unsuccessful polls it gives up and reports false (the caller flags an error
// and leaves its loop instead of hanging).
// ---------------------------------------------------------------------------
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i)
        if (mbar_try(bar, parity)) return true;
    return false;
}
// Same wait, but each try suspends the thread for up to `hint_ns` until the
// phase completes instead of returning at once: waiting warps then stop
// issuing polls that compete with the copies they wait for.  Bounded by
// kSleepLimit tries (seconds in total).
constexpr uint32_t kSleepLimit = 1u << 16;
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSleepLimit; ++i)
        if (mbar_try_sleep(bar, parity, 20000u)) return true;
    return false;
}
// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_pol(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                             uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;\n" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}
// TMA gather of four 128-byte row pieces: rows r0..r3, columns x..x+63 (bf16)
// of the 2-D tensor `tmap` (box 64 x 1, 128-byte swizzle) into 512
// consecutive shared bytes at `dst`, completing `bar`'s transaction count.
// x * 2 bytes must be a multiple of 16; the swizzle follows the shared
// address, so dst = region + 128 * row keeps the 128B-swizzle layout.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* tmap, int x, int r0, int r1, int r2, int r3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3, %4, %5, %6}], [%7];\n" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
        : "memory");
}
// TMA load of one 128-byte row piece: row y, columns x..x+63 (bf16) of the
// 2-D tensor `tmap` (box 64 x 1, 128-byte swizzle) into `dst`.
__device__ __forceinline__ void tma_load_row(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// TMA load of one box (the map's box: 64 bf16 columns x its rows) at column
// x, row y into consecutive 128-byte rows from `dst` (1024-byte aligned for
// the 128-byte swizzle).
__device__ __forceinline__ void tma_load_box(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
    tma_load_row(dst, tmap, x, y, bar);
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
// Shared -> global bulk copy (both addresses 16-byte aligned, bytes a
// multiple of 16), completed through the thread's bulk groups.
__device__ __forceinline__ void bulk_s2g(void* gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gdst), "r"(ssrc), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// the thread's committed bulk copies have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
// the thread's committed bulk copies are complete (their writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void named_bar(int id, int threads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace sgldev
