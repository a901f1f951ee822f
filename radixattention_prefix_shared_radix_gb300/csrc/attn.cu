// RadixAttention kernels for sm_103a and the GPU entry points of the C ABI.
//
// Decode ("SGLang 深度拆解" (chenxutan.com/d/5669.html) §3.2 PagedDecode and
// §4.1: one query token against the whole history, memory-bound) is split
// along the KV sequence into the planner's work items.  One CTA takes one
// (segment chunk, KV head, member block): it gathers the chunk's K/V rows
// through req_to_token ONCE into shared memory and runs every member
// request's query heads of that KV head against them ("computed once,
// referenced many times", oripoin.cn section "用基数树实现前缀复用").  Query
// rows (member x head) are packed 16 to a tensor-core tile.  Each item writes
// a normalised partial (O, LSE); a second kernel merges a request's partials
// by log-sum-exp with warp shuffles.
//
// Extend ("SGLang 深度拆解" §3.2 PagedPrefill; "SGLang 深度解读" section
// "5. Attention 层": the new tokens' K/V are in the pool before attention)
// packs (new token x query head of one KV head) rows 128 to a CTA and walks
// the cached prefix plus the causal part of the new block.
//
// Gathers: slots are random per token, so every K/V row (head_dim x 2 bytes,
// 16-byte aligned) is fetched with 16-byte cp.async into an XOR-swizzled
// shared-memory tile (conflict-free ldmatrix), three tiles in flight.
// Softmax runs in base 2 on scores pre-multiplied by sm_scale * log2(e);
// LSE is returned in natural log.  Slots outside the pool are skipped and
// flagged in the workspace error word; nothing traps.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.h"

namespace {

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

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte chunk c of row r in a swizzled tile of D-wide rows.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

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
template <int D, int NT>
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
            ldsm_x4_t(vbase + swz<D>(vr, dp * 2 + (lane >> 4)), b0, b1, b2, b3);
            mma16816(st.o[2 * dp], a, b0, b1);
            mma16816(st.o[2 * dp + 1], a, b2, b3);
        }
    }
}

// S[16 x 8*NT] = Q(m-tile, fragments qf) * K^T for the NT/2 16-row groups of
// KV rows starting at smem row krow0 of sK.
template <int D, int NT>
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
            ldsm_x4(kbase + swz<D>(kr, ks * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
            mma16816(s[2 * np], qf[ks], b0, b1);
            mma16816(s[2 * np + 1], qf[ks], b2, b3);
        }
    }
}

template <int D>
__device__ __forceinline__ void load_qfrag(uint32_t (&qf)[D / 16][4], const uint8_t* sQ, int row0, int lane) {
    const uint32_t qbase = smem_u32(sQ);
    const int r = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
        ldsm_x4(qbase + swz<D>(r, ks * 2 + (lane >> 4)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
}

// ---------------------------------------------------------------------------
// Decode partial kernel (bf16).  128 threads; up to 64 query rows per item.
// ---------------------------------------------------------------------------
template <int D>
constexpr int decode_smem_bytes() {
    return (64 + 2 * kStages * kTile) * D * 2;
}

template <int D>
__global__ void __launch_bounds__(128, 2)
    decode_partial_bf16(const bf16* __restrict__ q, const bf16* __restrict__ kp, const bf16* __restrict__ vp,
                        const int32_t* __restrict__ r2t, int64_t ld, const int32_t* __restrict__ seq_lens,
                        const sgl::DecItem* __restrict__ items, const int32_t* __restrict__ members,
                        float* __restrict__ po, float* __restrict__ plse, uint32_t* __restrict__ err, int Hq,
                        int Hkv, int G, int64_t num_slots, float scale_log2) {
    constexpr int CH = D / 8;           // 16-byte chunks per row
    constexpr int RB = D * 2;           // bytes per row
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* sQ = smem;
    uint8_t* sK = smem + 64 * RB;
    uint8_t* sV = sK + kStages * kTile * RB;

    const sgl::DecItem it = items[blockIdx.x];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rows = it.n_mem * G;
    int mt = (rows + 15) >> 4;
    const int mt_eff = mt == 3 ? 4 : mt;
    const int wpm = 4 / mt_eff;
    const int my_mt = warp / wpm, my_sub = warp % wpm;

    int kv_end = it.kv_end;
    const int rep_len = __ldg(seq_lens + it.rep_row);
    if (kv_end > rep_len) {
        if (tid == 0) atomicOr(err, 2u);
        kv_end = rep_len;
    }
    const int n_tok = kv_end - it.kv_begin;
    const int n_tiles = n_tok > 0 ? (n_tok + kTile - 1) / kTile : 0;

    // Q rows of the item: row = member * G + head-in-group.
    for (int i = tid; i < 64 * CH; i += 128) {
        const int r = i / CH, c = i % CH;
        const bf16* src = q;
        bool ok = r < rows;
        if (ok) {
            const int mem = __ldg(members + it.mem_begin + r / G);
            src = q + ((int64_t)mem * Hq + it.kvh * G + r % G) * D + c * 8;
        }
        cp_async16(smem_u32(sQ) + swz<D>(r, c), src, ok);
    }
    cp_async_commit();

    // KV gather: thread -> (tile row tid/2, half of the chunks).
    const int grow = tid >> 1, gc0 = (tid & 1) * (CH / 2);
    auto slot_at = [&](int tile) -> int64_t {
        const int rel = tile * kTile + grow;
        if (tile >= n_tiles || rel >= n_tok) return -1;
        return load_slot(r2t, ld, it.rep_row, it.kv_begin + rel, num_slots, err);
    };
    auto issue = [&](int tile, int64_t slot) {
        const int stg = tile % kStages;
        const int sr = stg * kTile + grow;
        const bool ok = slot >= 0;
        const int64_t off = ok ? (slot * Hkv + it.kvh) * D : 0;
#pragma unroll
        for (int c = gc0; c < gc0 + CH / 2; ++c) {
            cp_async16(smem_u32(sK) + swz<D>(sr, c), kp + off + c * 8, ok);
            cp_async16(smem_u32(sV) + swz<D>(sr, c), vp + off + c * 8, ok);
        }
    };
#pragma unroll
    for (int t = 0; t < kStages - 1; ++t) {
        if (t < n_tiles) issue(t, slot_at(t));
        cp_async_commit();
    }
    int64_t next_slot = slot_at(kStages - 1);

    cp_async_wait<kStages - 1>();
    __syncthreads();
    uint32_t qf[D / 16][4];
    load_qfrag<D>(qf, sQ, (my_mt < mt ? my_mt : 0) * 16, lane);

    WarpState<D> st;
    st.init();
    for (int tile = 0; tile < n_tiles; ++tile) {
        const int nt = tile + kStages - 1;
        if (nt < n_tiles) issue(nt, next_slot);
        cp_async_commit();
        next_slot = slot_at(nt + 1);
        cp_async_wait<kStages - 1>();
        __syncthreads();
        const int stg = tile % kStages;
        if (my_mt < mt) {
            for (int k = my_sub; k < kTile / 16; k += wpm) {
                const int tok0 = tile * kTile + k * 16;
                if (tok0 >= n_tok) break;
                float s[2][4];
                qk<D, 2>(s, qf, sK, stg * kTile + k * 16, lane);
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int tok = tok0 + n * 8 + 2 * (lane & 3) + (e & 1);
                        s[n][e] = tok < n_tok ? s[n][e] * scale_log2 : -INFINITY;
                    }
                softmax_pv<D, 2>(st, s, sV, stg * kTile + k * 16, lane);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    __syncthreads();

    // Combine the warps that share an m-tile, normalise, write the partials.
    float* sO = reinterpret_cast<float*>(sK);                 // [4][16][D]
    float* sM = reinterpret_cast<float*>(sV);                 // [4][16]
    float* sL = sM + 64;
    const int g = lane >> 2, t4 = lane & 3;
    st.l[0] = quad_sum(st.l[0]);
    st.l[1] = quad_sum(st.l[1]);
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        float* r0 = sO + (warp * 16 + g) * D + n * 8 + 2 * t4;
        float* r1 = sO + (warp * 16 + g + 8) * D + n * 8 + 2 * t4;
        r0[0] = st.o[n][0];
        r0[1] = st.o[n][1];
        r1[0] = st.o[n][2];
        r1[1] = st.o[n][3];
    }
    if (t4 == 0) {
        sM[warp * 16 + g] = st.m[0];
        sM[warp * 16 + g + 8] = st.m[1];
        sL[warp * 16 + g] = st.l[0];
        sL[warp * 16 + g + 8] = st.l[1];
    }
    __syncthreads();
    for (int idx = tid; idx < rows * (D / 4); idx += 128) {
        const int r = idx / (D / 4), c4 = idx % (D / 4);
        const int mtile = r >> 4, i = r & 15;
        float M = -INFINITY;
        for (int w = mtile * wpm; w < (mtile + 1) * wpm; ++w) M = fmaxf(M, sM[w * 16 + i]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
        if (M != -INFINITY) {
            for (int w = mtile * wpm; w < (mtile + 1) * wpm; ++w) {
                const float wt = exp2f(sM[w * 16 + i] - M);
                const float4 v = *reinterpret_cast<const float4*>(sO + (w * 16 + i) * D + c4 * 4);
                acc.x += wt * v.x;
                acc.y += wt * v.y;
                acc.z += wt * v.z;
                acc.w += wt * v.w;
                L += wt * sL[w * 16 + i];
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        float4 out = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        const int64_t prow = (int64_t)it.partial_base + r;
        *reinterpret_cast<float4*>(po + prow * D + c4 * 4) = out;
        if (c4 == 0) plse[prow] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
}

// ---------------------------------------------------------------------------
// Decode partial kernel (fp32, CUDA cores, no tensor cores): one warp per
// query row of the item, lanes split head_dim; exact fp32 FFMA dot products.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128)
    decode_partial_f32(const float* __restrict__ q, const float* __restrict__ kp, const float* __restrict__ vp,
                       const int32_t* __restrict__ r2t, int64_t ld, const int32_t* __restrict__ seq_lens,
                       const sgl::DecItem* __restrict__ items, const int32_t* __restrict__ members,
                       float* __restrict__ po, float* __restrict__ plse, uint32_t* __restrict__ err, int Hq, int Hkv,
                       int G, int64_t num_slots, float scale_log2) {
    constexpr int E = D / 32;
    const sgl::DecItem it = items[blockIdx.x];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rows = it.n_mem * G;
    int kv_end = it.kv_end;
    const int rep_len = __ldg(seq_lens + it.rep_row);
    if (kv_end > rep_len) {
        if (threadIdx.x == 0) atomicOr(err, 2u);
        kv_end = rep_len;
    }
    for (int r = warp; r < rows; r += 4) {
        const int mem = __ldg(members + it.mem_begin + r / G);
        const float* qr = q + ((int64_t)mem * Hq + it.kvh * G + r % G) * D + lane * E;
        float qv[E], o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            qv[e] = qr[e];
            o[e] = 0.f;
        }
        float m = -INFINITY, l = 0.f;
        for (int pos = it.kv_begin; pos < kv_end; ++pos) {
            const int64_t slot = load_slot(r2t, ld, it.rep_row, pos, num_slots, err);
            if (slot < 0) continue;
            const float* kr = kp + (slot * Hkv + it.kvh) * D + lane * E;
            const float* vr = vp + (slot * Hkv + it.kvh) * D + lane * E;
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) dot = fmaf(qv[e], kr[e], dot);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            const float s = dot * scale_log2;
            const float mn = fmaxf(m, s);
            const float a = exp2f(m - mn), p = exp2f(s - mn);
            l = l * a + p;
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = fmaf(p, vr[e], o[e] * a);
            m = mn;
        }
        const int64_t prow = (int64_t)it.partial_base + r;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) po[prow * D + lane * E + e] = o[e] * inv;
        if (lane == 0) plse[prow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
}

// ---------------------------------------------------------------------------
// Merge: one warp per (request, query head); log-sum-exp over its partials.
// ---------------------------------------------------------------------------
template <typename OutT>
__device__ __forceinline__ void store_out(OutT* p, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* p, float v) {
    *p = v;
}
template <>
__device__ __forceinline__ void store_out<bf16>(bf16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

template <typename OutT, int D>
__global__ void __launch_bounds__(128)
    decode_merge(const float* __restrict__ po, const float* __restrict__ plse, const int32_t* __restrict__ mptr,
                 const sgl::MergeEnt* __restrict__ ment, OutT* __restrict__ o, float* __restrict__ lse, int B, int Hq,
                 int G) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int idx = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (idx >= B * Hq) return;
    const int r = idx / Hq, h = idx % Hq, g = h / G, j = h % G;
    const int e0 = __ldg(mptr + r), e1 = __ldg(mptr + r + 1);
    float M = -INFINITY;
    for (int e = e0 + lane; e < e1; e += 32) {
        const sgl::MergeEnt me = ment[e];
        M = fmaxf(M, plse[me.pbase + g * me.gstride + j]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[E];
#pragma unroll
    for (int k = 0; k < E; ++k) acc[k] = 0.f;
    float L = 0.f;
    if (M != -INFINITY) {
        for (int e = e0; e < e1; ++e) {
            const sgl::MergeEnt me = ment[e];
            const int64_t prow = me.pbase + g * me.gstride + j;
            const float w = exp2f((plse[prow] - M) * kLog2e);
            L += w;
            const float* src = po + prow * D + lane * E;
#pragma unroll
            for (int k = 0; k < E; ++k) acc[k] = fmaf(w, src[k], acc[k]);
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    OutT* dst = o + ((int64_t)r * Hq + h) * D + lane * E;
#pragma unroll
    for (int k = 0; k < E; ++k) store_out<OutT>(dst + k, acc[k] * inv);
    if (lane == 0) lse[(int64_t)r * Hq + h] = L > 0.f ? M + logf(L) : -INFINITY;
}

// ---------------------------------------------------------------------------
// Extend kernel (bf16).  256 threads = 8 warps x 16 rows = 128 query rows per
// CTA: (128 / G) new tokens x G query heads of one KV head.
// ---------------------------------------------------------------------------
template <int D>
constexpr int extend_smem_bytes() {
    return (128 + 2 * kStages * kTile) * D * 2;
}

// Request of tile `t` (tiles of tq new tokens, request by request), its
// first tile index and its first q row, by a scan over extend_lens.
__device__ __forceinline__ void find_tile(const int32_t* ext, int B, int tq, int t, int* req, int* tile0, int* qoff) {
    int acc_t = 0, acc_q = 0;
    for (int r = 0; r < B; ++r) {
        const int e = __ldg(ext + r);
        const int nt = (e + tq - 1) / tq;
        if (t < acc_t + nt) {
            *req = r;
            *tile0 = acc_t;
            *qoff = acc_q;
            return;
        }
        acc_t += nt;
        acc_q += e;
    }
    *req = -1;
}

template <int D>
__global__ void __launch_bounds__(256, 1)
    extend_bf16(const bf16* __restrict__ qn, const bf16* __restrict__ kp, const bf16* __restrict__ vp,
                const int32_t* __restrict__ r2t, int64_t ld, const int32_t* __restrict__ prefix_lens,
                const int32_t* __restrict__ extend_lens, bf16* __restrict__ o, float* __restrict__ lse,
                uint32_t* __restrict__ err, int B, int Hq, int Hkv, int G, int64_t num_slots, int64_t n_rows,
                float scale_log2) {
    constexpr int CH = D / 8;
    constexpr int RB = D * 2;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* sQ = smem;
    uint8_t* sK = smem + 128 * RB;
    uint8_t* sV = sK + kStages * kTile * RB;
    __shared__ int s_req, s_tile0, s_qoff;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tq = 128 / G;
    const int kvh = blockIdx.y;
    if (tid == 0) find_tile(extend_lens, B, tq, blockIdx.x, &s_req, &s_tile0, &s_qoff);
    __syncthreads();
    const int req = s_req;
    if (req < 0) return;
    const int pre = __ldg(prefix_lens + req), ext = __ldg(extend_lens + req);
    const int t0 = (blockIdx.x - s_tile0) * tq;             // first new token of the tile
    const int ntok = min(tq, ext - t0);
    // the device lengths must agree with the host copies the grid was sized from
    if (pre < 0 || ntok <= 0 || (int64_t)pre + ext > ld || (int64_t)s_qoff + t0 + ntok > n_rows) {
        if (tid == 0) atomicOr(err, 2u);
        return;
    }
    const int rows = ntok * G;
    const int kv_len = pre + t0 + ntok;                      // positions [0, kv_len)
    const int n_tiles = (kv_len + kTile - 1) / kTile;
    const int64_t qrow0 = (int64_t)s_qoff + t0;

    for (int i = tid; i < 128 * CH; i += 256) {
        const int r = i / CH, c = i % CH;
        const bool ok = r < rows;
        const bf16* src = ok ? qn + ((qrow0 + r / G) * Hq + kvh * G + r % G) * D + c * 8 : qn;
        cp_async16(smem_u32(sQ) + swz<D>(r, c), src, ok);
    }
    cp_async_commit();

    // gather: 4 threads per KV row, CH/4 chunks each
    const int grow = tid >> 2, gc0 = (tid & 3) * (CH / 4);
    auto slot_at = [&](int tile) -> int64_t {
        const int pos = tile * kTile + grow;
        if (tile >= n_tiles || pos >= kv_len) return -1;
        return load_slot(r2t, ld, req, pos, num_slots, err);
    };
    auto issue = [&](int tile, int64_t slot) {
        const int sr = (tile % kStages) * kTile + grow;
        const bool ok = slot >= 0;
        const int64_t off = ok ? (slot * Hkv + kvh) * D : 0;
#pragma unroll
        for (int c = gc0; c < gc0 + CH / 4; ++c) {
            cp_async16(smem_u32(sK) + swz<D>(sr, c), kp + off + c * 8, ok);
            cp_async16(smem_u32(sV) + swz<D>(sr, c), vp + off + c * 8, ok);
        }
    };
#pragma unroll
    for (int t = 0; t < kStages - 1; ++t) {
        if (t < n_tiles) issue(t, slot_at(t));
        cp_async_commit();
    }
    int64_t next_slot = slot_at(kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncthreads();
    uint32_t qf[D / 16][4];
    load_qfrag<D>(qf, sQ, warp * 16, lane);

    // causal limits of this thread's two rows (g and g+8 of the warp's m-tile)
    const int g = lane >> 2, t4 = lane & 3;
    const int lim0 = pre + t0 + (warp * 16 + g) / G;
    const int lim1 = pre + t0 + (warp * 16 + g + 8) / G;
    const bool warp_live = warp * 16 < rows;

    WarpState<D> st;
    st.init();
    for (int tile = 0; tile < n_tiles; ++tile) {
        const int nt = tile + kStages - 1;
        if (nt < n_tiles) issue(nt, next_slot);
        cp_async_commit();
        next_slot = slot_at(nt + 1);
        cp_async_wait<kStages - 1>();
        __syncthreads();
        if (warp_live) {
            const int stg = tile % kStages;
            float s[kTile / 8][4];
            qk<D, kTile / 8>(s, qf, sK, stg * kTile, lane);
            const int pos0 = tile * kTile;
            const bool need_mask = pos0 + kTile - 1 > pre + t0;
#pragma unroll
            for (int n = 0; n < kTile / 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int pos = pos0 + n * 8 + 2 * t4 + (e & 1);
                    const int lim = e < 2 ? lim0 : lim1;
                    s[n][e] = (!need_mask || pos <= lim) ? s[n][e] * scale_log2 : -INFINITY;
                }
            softmax_pv<D, kTile / 8>(st, s, sV, stg * kTile, lane);
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    if (!warp_live) return;
    const float l0 = quad_sum(st.l[0]), l1 = quad_sum(st.l[1]);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const int r0 = warp * 16 + g, r1 = r0 + 8;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        if (r0 < rows) {
            bf16* dst = o + ((qrow0 + r0 / G) * Hq + kvh * G + r0 % G) * D + n * 8 + 2 * t4;
            *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(st.o[n][0] * inv0, st.o[n][1] * inv0);
        }
        if (r1 < rows) {
            bf16* dst = o + ((qrow0 + r1 / G) * Hq + kvh * G + r1 % G) * D + n * 8 + 2 * t4;
            *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(st.o[n][2] * inv1, st.o[n][3] * inv1);
        }
    }
    if (t4 == 0) {
        if (r0 < rows) lse[(qrow0 + r0 / G) * Hq + kvh * G + r0 % G] = l0 > 0.f ? (st.m[0] + log2f(l0)) * kLn2 : -INFINITY;
        if (r1 < rows) lse[(qrow0 + r1 / G) * Hq + kvh * G + r1 % G] = l1 > 0.f ? (st.m[1] + log2f(l1)) * kLn2 : -INFINITY;
    }
}

// ---------------------------------------------------------------------------
// Extend (fp32, CUDA cores): one warp per (new token, query head).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128)
    extend_f32(const float* __restrict__ qn, const float* __restrict__ kp, const float* __restrict__ vp,
               const int32_t* __restrict__ r2t, int64_t ld, const int32_t* __restrict__ prefix_lens,
               const int32_t* __restrict__ extend_lens, float* __restrict__ o, float* __restrict__ lse,
               uint32_t* __restrict__ err, int B, int Hq, int Hkv, int G, int64_t num_slots, int64_t n_rows,
               float scale_log2) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);   // (new row, head)
    const int h = (int)(w % Hq);
    const int64_t nrow = w / Hq;
    if (nrow >= n_rows) return;
    int req = -1, acc = 0;
    for (int r = 0; r < B; ++r) {
        const int e = __ldg(extend_lens + r);
        if (nrow < acc + e) {
            req = r;
            break;
        }
        acc += e;
    }
    if (req < 0) return;
    const int i = (int)(nrow - acc);
    const int pre = __ldg(prefix_lens + req);
    if (pre < 0 || (int64_t)pre + __ldg(extend_lens + req) > ld) {
        if (lane == 0) atomicOr(err, 2u);
        return;
    }
    const int lim = pre + i;
    const int kvh = h / G;
    const float* qr = qn + (nrow * Hq + h) * D + lane * E;
    float qv[E], ov[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qv[e] = qr[e];
        ov[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int pos = 0; pos <= lim; ++pos) {
        const int64_t slot = load_slot(r2t, ld, req, pos, num_slots, err);
        if (slot < 0) continue;
        const float* kr = kp + (slot * Hkv + kvh) * D + lane * E;
        const float* vr = vp + (slot * Hkv + kvh) * D + lane * E;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot = fmaf(qv[e], kr[e], dot);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float s = dot * scale_log2;
        const float mn = fmaxf(m, s);
        const float a = exp2f(m - mn), p = exp2f(s - mn);
        l = l * a + p;
#pragma unroll
        for (int e = 0; e < E; ++e) ov[e] = fmaf(p, vr[e], ov[e] * a);
        m = mn;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[(nrow * Hq + h) * D + lane * E + e] = ov[e] * inv;
    if (lane == 0) lse[nrow * Hq + h] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
thread_local int t_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SGL_OK;
    t_last_cuda_error = static_cast<int>(e);
    return SGL_ERR_CUDA;
}

template <typename K>
cudaError_t allow_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

float scale_log2_of(const sgl_attn_params* p) {
    const float sc = p->sm_scale > 0.f ? p->sm_scale : 1.0f / std::sqrt(static_cast<float>(p->head_dim));
    return sc * kLog2e;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <int D>
int launch_decode(const sgl_plan* plan, const void* q, const void* kp, const void* vp, const int32_t* r2t,
                  int64_t ld, const int32_t* seq_lens, void* o, float* lse, unsigned char* ws, cudaStream_t s) {
    const sgl_attn_params& p = plan->params;
    const auto* items = reinterpret_cast<const sgl::DecItem*>(ws + plan->off_items);
    const auto* members = reinterpret_cast<const int32_t*>(ws + plan->off_members);
    const auto* mptr = reinterpret_cast<const int32_t*>(ws + plan->off_mptr);
    const auto* ment = reinterpret_cast<const sgl::MergeEnt*>(ws + plan->off_ment);
    float* plse = reinterpret_cast<float*>(ws + plan->off_plse);
    float* po = reinterpret_cast<float*>(ws + plan->off_po);
    uint32_t* err = reinterpret_cast<uint32_t*>(ws);
    const float sl2 = scale_log2_of(&p);
    const int Hq = p.num_qo_heads, Hkv = p.num_kv_heads, G = plan->G, B = p.batch;
    if (p.dtype == SGL_DTYPE_BF16) {
        static bool once = [] { return allow_smem(decode_partial_bf16<D>, decode_smem_bytes<D>()) == cudaSuccess; }();
        if (!once) return cuda_status(cudaGetLastError());
        if (plan->n_items > 0)
            decode_partial_bf16<D><<<plan->n_items, 128, decode_smem_bytes<D>(), s>>>(
                static_cast<const bf16*>(q), static_cast<const bf16*>(kp), static_cast<const bf16*>(vp), r2t, ld,
                seq_lens, items, members, po, plse, err, Hq, Hkv, G, p.num_slots, sl2);
        if (B > 0)
            decode_merge<bf16, D><<<(B * Hq + 3) / 4, 128, 0, s>>>(po, plse, mptr, ment, static_cast<bf16*>(o), lse,
                                                                   B, Hq, G);
    } else {
        if (plan->n_items > 0)
            decode_partial_f32<D><<<plan->n_items, 128, 0, s>>>(
                static_cast<const float*>(q), static_cast<const float*>(kp), static_cast<const float*>(vp), r2t, ld,
                seq_lens, items, members, po, plse, err, Hq, Hkv, G, p.num_slots, sl2);
        if (B > 0)
            decode_merge<float, D><<<(B * Hq + 3) / 4, 128, 0, s>>>(po, plse, mptr, ment, static_cast<float*>(o),
                                                                    lse, B, Hq, G);
    }
    return cuda_status(cudaGetLastError());
}

template <int D>
int launch_extend(const sgl_attn_params* p, const void* q, const void* kp, const void* vp, const int32_t* r2t,
                  int64_t ld, const int32_t* pre, const int32_t* ext, void* o, float* lse, uint32_t* err,
                  cudaStream_t s) {
    const int Hq = p->num_qo_heads, Hkv = p->num_kv_heads, G = Hq / Hkv, B = p->batch;
    const float sl2 = scale_log2_of(p);
    int64_t total_rows = 0, tiles = 0;
    const int tq = 128 / G;
    for (int r = 0; r < B; ++r) {
        total_rows += p->host_extend_lens[r];
        tiles += (p->host_extend_lens[r] + tq - 1) / tq;
    }
    if (total_rows == 0) return SGL_OK;
    if (p->dtype == SGL_DTYPE_BF16) {
        static bool once = [] { return allow_smem(extend_bf16<D>, extend_smem_bytes<D>()) == cudaSuccess; }();
        if (!once) return cuda_status(cudaGetLastError());
        if (tiles > INT32_MAX) return SGL_ERR_UNSUPPORTED;
        dim3 grid(static_cast<unsigned>(tiles), Hkv);
        extend_bf16<D><<<grid, 256, extend_smem_bytes<D>(), s>>>(
            static_cast<const bf16*>(q), static_cast<const bf16*>(kp), static_cast<const bf16*>(vp), r2t, ld, pre,
            ext, static_cast<bf16*>(o), lse, err, B, Hq, Hkv, G, p->num_slots, total_rows, sl2);
    } else {
        const int64_t warps = total_rows * Hq;
        if ((warps + 3) / 4 > INT32_MAX) return SGL_ERR_UNSUPPORTED;
        extend_f32<D><<<static_cast<unsigned>((warps + 3) / 4), 128, 0, s>>>(
            static_cast<const float*>(q), static_cast<const float*>(kp), static_cast<const float*>(vp), r2t, ld, pre,
            ext, static_cast<float*>(o), lse, err, B, Hq, Hkv, G, p->num_slots, total_rows, sl2);
    }
    return cuda_status(cudaGetLastError());
}

}  // namespace

namespace sgl {
int check_params(const sgl_attn_params* p);
void set_cuda_error(int err) { t_last_cuda_error = err; }
}  // namespace sgl

extern "C" {

int sgl_last_cuda_error(void) { return t_last_cuda_error; }

int sgl_plan_upload(const sgl_plan* plan, void* workspace, size_t ws_bytes, sgl_stream_t stream) {
    if (!plan || !workspace) return SGL_ERR_INVALID_ARG;
    if (!aligned(workspace, sgl::kWsAlign) || ws_bytes < plan->workspace_bytes) return SGL_ERR_WORKSPACE;
    return cuda_status(cudaMemcpyAsync(workspace, plan->blob, plan->tables_bytes, cudaMemcpyHostToDevice,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int sgl_decode_attn(const void* q, const void* k_pool, const void* v_pool, const int32_t* req_to_token, int64_t ld,
                    const int32_t* seq_lens, const sgl_plan* plan, void* o, float* lse, void* workspace,
                    size_t ws_bytes, sgl_stream_t stream) {
    if (!plan) return SGL_ERR_INVALID_ARG;
    const int32_t B = plan->params.batch;
    if (B > 0 && (!q || !o || !lse || !seq_lens)) return SGL_ERR_INVALID_ARG;
    if (plan->n_items > 0 && (!k_pool || !v_pool || !req_to_token || ld < plan->max_pos)) return SGL_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, sgl::kWsAlign) || ws_bytes < plan->workspace_bytes)
        return SGL_ERR_WORKSPACE;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o, 16))
        return SGL_ERR_INVALID_ARG;
    auto* ws = static_cast<unsigned char*>(workspace);
    auto s = reinterpret_cast<cudaStream_t>(stream);
    if (plan->params.head_dim == 128) return launch_decode<128>(plan, q, k_pool, v_pool, req_to_token, ld, seq_lens, o, lse, ws, s);
    return launch_decode<64>(plan, q, k_pool, v_pool, req_to_token, ld, seq_lens, o, lse, ws, s);
}

int sgl_extend_attn(const void* q_new, const void* k_pool, const void* v_pool, const int32_t* req_to_token,
                    int64_t ld, const int32_t* prefix_lens, const int32_t* extend_lens, const sgl_attn_params* params,
                    void* o, float* lse, void* workspace, size_t ws_bytes, sgl_stream_t stream) {
    int st = sgl::check_params(params);
    if (st) return st;
    const int32_t B = params->batch;
    if (B > 0 && (!params->host_extend_lens || !params->host_prefix_lens || !prefix_lens || !extend_lens))
        return SGL_ERR_INVALID_ARG;
    int64_t rows = 0;
    for (int32_t r = 0; r < B; ++r) {
        if (params->host_extend_lens[r] < 0 || params->host_prefix_lens[r] < 0) return SGL_ERR_INVALID_ARG;
        if ((int64_t)params->host_prefix_lens[r] + params->host_extend_lens[r] > ld) return SGL_ERR_INVALID_ARG;
        rows += params->host_extend_lens[r];
    }
    if (rows > 0 && (!q_new || !k_pool || !v_pool || !req_to_token || !o || !lse)) return SGL_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, sgl::kWsAlign) || ws_bytes < sgl::kWsAlign) return SGL_ERR_WORKSPACE;
    if (!aligned(q_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o, 16))
        return SGL_ERR_INVALID_ARG;
    auto s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t* err = static_cast<uint32_t*>(workspace);
    if (params->head_dim == 128)
        return launch_extend<128>(params, q_new, k_pool, v_pool, req_to_token, ld, prefix_lens, extend_lens, o, lse,
                                  err, s);
    return launch_extend<64>(params, q_new, k_pool, v_pool, req_to_token, ld, prefix_lens, extend_lens, o, lse, err,
                             s);
}

int sgl_check(void* workspace, sgl_stream_t stream) {
    if (!workspace) return SGL_ERR_INVALID_ARG;
    auto s = reinterpret_cast<cudaStream_t>(stream);
    int st = cuda_status(cudaStreamSynchronize(s));
    if (st) return st;
    uint32_t word = 0;
    st = cuda_status(cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost));
    if (st) return st;
    if (word == 0) return SGL_OK;
    st = cuda_status(cudaMemset(workspace, 0, sizeof(word)));
    if (st) return st;
    return SGL_ERR_BOUNDS;
}

}  // extern "C"
