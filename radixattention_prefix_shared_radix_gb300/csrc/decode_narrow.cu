// Decode for narrow work items (at most 8 query rows per KV head: one
// request's G query heads, or a few members of a small group) and the
// log-sum-exp merge of all decode partials.
//
// One warp per work item; no shared memory and no block-wide barriers, so an
// SM keeps ~14 independent warps with their K/V loads in flight (random
// 256-byte rows of the slot-major pool gather at >90% of a sequential read
// when enough loads are outstanding).
//
// Tensor-core formulation (mma.sync m16n8k16, bf16 in, fp32 accumulate), per
// 16 KV positions:
//   S^T [16 pos x 8 rows]  = K [16 x d] . Q^T [d x 8 rows]
//   O^T [d x 8 rows]      += V^T [d x 16 pos] . P^T [16 pos x 8 rows]
// Query rows sit in the MMA's N dimension (8 wide), so a request's 4 query
// heads waste half an n-tile instead of 3/4 of an m-tile.  P^T goes from the
// accumulator layout to the B-operand layout with movmatrix (8x8 transpose in
// registers).  Operands come straight from global memory into registers:
//   * the head dimension of K and Q is permuted so that lane (g, t) of an
//     m16n8k16 fragment needs the 16-byte chunks t, t+4, t+8, ... of the row
//     (a permutation of the summation index leaves Q.K unchanged), so the 4
//     lanes of a row read 64 contiguous bytes per instruction;
//   * the head dimension of V (and so of O^T) is permuted so that lane
//     (g, t) needs chunks g, g+8, ... of four V rows (8 lanes read 128
//     contiguous bytes of a row per instruction); the permutation is undone
//     when O is written.
// Softmax is online in base 2 on scores pre-scaled by sm_scale * log2(e).
// Every work item writes normalised partial rows (O fp32, LSE natural log);
// decode_merge combines a request's partials per KV head.

#include "device_common.cuh"

namespace sgl {

namespace {

using namespace sgldev;

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

template <int D>
__global__ void __launch_bounds__(128)
    decode_narrow_bf16(const bf16* __restrict__ q, const bf16* __restrict__ kp, const bf16* __restrict__ vp,
                       const int32_t* __restrict__ r2t, int64_t ld, const int32_t* __restrict__ seq_lens,
                       const DecItem* __restrict__ items, int n_items, const int32_t* __restrict__ members,
                       float* __restrict__ po, float* __restrict__ plse, uint32_t* __restrict__ err, int Hq, int Hkv,
                       int G, int64_t num_slots, float scale_log2) {
    constexpr int KW = D / 8;    // 32-bit words of K (and Q) a lane holds per row: chunks t + 4c
    constexpr int VW = D / 16;   // words of V a lane holds per row: chunks g + 8c
    constexpr int MT = D / 16;   // m-tiles of O^T (16 head-dim rows each)
    const int lane = threadIdx.x & 31;
    const int wi = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (wi >= n_items) return;
    const DecItem it = items[wi];
    const int g = lane >> 2, t = lane & 3;
    const int rows = it.n_mem * G;

    int e = it.kv_end;
    const int rep_len = __ldg(seq_lens + it.rep_row);
    if (e > rep_len) {
        if (lane == 0) atomicOr(err, 2u);
        e = rep_len;
    }
    const int b = it.kv_begin;

    // Q^T fragments: row g (zero if padding), chunks t + 4c
    uint32_t qw[KW];
    {
        const bool ok = g < rows;
        const bf16* qrow = q;
        if (ok) {
            const int mem = __ldg(members + it.mem_begin + g / G);
            qrow = q + ((int64_t)mem * Hq + it.kvh * G + g % G) * D;
        }
#pragma unroll
        for (int c = 0; c < KW / 4; ++c) {
            uint4 v = ok ? __ldg(reinterpret_cast<const uint4*>(qrow) + t + 4 * c) : make_uint4(0, 0, 0, 0);
            qw[4 * c] = v.x;
            qw[4 * c + 1] = v.y;
            qw[4 * c + 2] = v.z;
            qw[4 * c + 3] = v.w;
        }
    }

    float o[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows 2t, 2t+1

    const int32_t* trow = r2t + (int64_t)it.rep_row * ld;
    // slots of positions p0 + lane (lanes 0..15), loaded one step ahead
    int32_t raw = (lane < 16 && b + lane < e) ? __ldg(trow + b + lane) : -1;
    for (int p0 = b; p0 < e; p0 += 16) {
        int32_t sl = raw;
        raw = (lane < 16 && p0 + 16 + lane < e) ? __ldg(trow + p0 + 16 + lane) : -1;
        if (lane < 16 && p0 + lane < e && (sl < 0 || sl >= num_slots)) {
            atomicOr(err, 1u);
            sl = -1;
        }
        const int32_t sk0 = __shfl_sync(0xffffffffu, sl, g), sk1 = __shfl_sync(0xffffffffu, sl, g + 8);
        const int32_t sv0 = __shfl_sync(0xffffffffu, sl, 2 * t), sv1 = __shfl_sync(0xffffffffu, sl, 2 * t + 1);
        const int32_t sv2 = __shfl_sync(0xffffffffu, sl, 2 * t + 8), sv3 = __shfl_sync(0xffffffffu, sl, 2 * t + 9);

        // K rows g, g+8: chunks t + 4c
        uint32_t k0[KW], k1[KW];
        {
            const uint4* r0 = reinterpret_cast<const uint4*>(kp + ((int64_t)(sk0 < 0 ? 0 : sk0) * Hkv + it.kvh) * D) + t;
            const uint4* r1 = reinterpret_cast<const uint4*>(kp + ((int64_t)(sk1 < 0 ? 0 : sk1) * Hkv + it.kvh) * D) + t;
#pragma unroll
            for (int c = 0; c < KW / 4; ++c) {
                uint4 a = sk0 >= 0 ? __ldg(r0 + 4 * c) : make_uint4(0, 0, 0, 0);
                uint4 bb = sk1 >= 0 ? __ldg(r1 + 4 * c) : make_uint4(0, 0, 0, 0);
                k0[4 * c] = a.x;
                k0[4 * c + 1] = a.y;
                k0[4 * c + 2] = a.z;
                k0[4 * c + 3] = a.w;
                k1[4 * c] = bb.x;
                k1[4 * c + 1] = bb.y;
                k1[4 * c + 2] = bb.z;
                k1[4 * c + 3] = bb.w;
            }
        }
        // V rows 2t, 2t+1, 2t+8, 2t+9: chunks g + 8c
        uint32_t v[4][VW];
        {
            const int32_t sv[4] = {sv0, sv1, sv2, sv3};
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const uint4* r =
                    reinterpret_cast<const uint4*>(vp + ((int64_t)(sv[rr] < 0 ? 0 : sv[rr]) * Hkv + it.kvh) * D) + g;
#pragma unroll
                for (int c = 0; c < VW / 4; ++c) {
                    uint4 a = sv[rr] >= 0 ? __ldg(r + 8 * c) : make_uint4(0, 0, 0, 0);
                    v[rr][4 * c] = a.x;
                    v[rr][4 * c + 1] = a.y;
                    v[rr][4 * c + 2] = a.z;
                    v[rr][4 * c + 3] = a.w;
                }
            }
        }

        // S^T = K Q^T: accumulator (pos g, rows 2t, 2t+1), (pos g+8, rows 2t, 2t+1)
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t a[4] = {k0[2 * ks], k1[2 * ks], k0[2 * ks + 1], k1[2 * ks + 1]};
            mma16816(s, a, qw[2 * ks], qw[2 * ks + 1]);
        }
        const bool ok0 = p0 + g < e, ok1 = p0 + g + 8 < e;
        s[0] = ok0 ? s[0] * scale_log2 : -INFINITY;
        s[1] = ok0 ? s[1] * scale_log2 : -INFINITY;
        s[2] = ok1 ? s[2] * scale_log2 : -INFINITY;
        s[3] = ok1 ? s[3] * scale_log2 : -INFINITY;
        float x0 = fmaxf(s[0], s[2]), x1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
        }
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
        const float al0 = exp2f(m0 - u0), al1 = exp2f(m1 - u1);
        m0 = n0;
        m1 = n1;
        const float p00 = exp2f(s[0] - u0), p01 = exp2f(s[1] - u1);
        const float p10 = exp2f(s[2] - u0), p11 = exp2f(s[3] - u1);
        l0 = l0 * al0 + p00 + p10;
        l1 = l1 * al1 + p01 + p11;
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            o[i][0] *= al0;
            o[i][1] *= al1;
            o[i][2] *= al0;
            o[i][3] *= al1;
        }
        // P^T as the B operand: (pos 2t, 2t+1; row g) and (pos 2t+8, 2t+9; row g)
        const uint32_t pb0 = movtrans(pack_bf16(p00, p01));
        const uint32_t pb1 = movtrans(pack_bf16(p10, p11));
        // O^T += V^T P^T; m-tile i = 4c + u uses word i of the lane's V chunks:
        // its rows g, g+8 are head-dim elements 8g + 64c + 2u and that + 1
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const uint32_t a[4] = {__byte_perm(v[0][i], v[1][i], 0x5410), __byte_perm(v[0][i], v[1][i], 0x7632),
                                   __byte_perm(v[2][i], v[3][i], 0x5410), __byte_perm(v[2][i], v[3][i], 0x7632)};
            mma16816(o[i], a, pb0, pb1);
        }
    }

    // row sums over the 8 lanes of each t, normalise, write rows 2t, 2t+1
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = 2 * t + h;
        if (r >= rows) continue;
        const float inv = h ? i1 : i0;
        float* dst = po + ((int64_t)it.partial_base + r) * D + 8 * g;
#pragma unroll
        for (int c = 0; c < MT / 4; ++c) {
            // elements 8g + 64c .. +7 = m-tiles 4c .. 4c+3 (two elements each)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i0 = 4 * c + 2 * hh;
                *reinterpret_cast<float4*>(dst + 64 * c + 4 * hh) = make_float4(
                    o[i0][h] * inv, o[i0][2 + h] * inv, o[i0 + 1][h] * inv, o[i0 + 1][2 + h] * inv);
            }
        }
        if (g == 0) {
            const float mm = h ? m1 : m0, ll = h ? l1 : l0;
            plse[(int64_t)it.partial_base + r] = ll > 0.f ? (mm + log2f(ll)) * kLn2 : -INFINITY;
        }
    }
}

// Merge: one CTA per (request, KV head).  The partial rows and LSEs of all
// the request's entries for the G heads are staged in shared memory in one
// parallel sweep; then thread u (query head j = u / (D/4), four head-dim
// elements) forms the LSE-weighted sum with its loads issued four at a time.
constexpr int kMergeStage = 2048;   // staged (entry, head) pairs; more fall back to direct loads

template <typename OutT, int D>
__global__ void __launch_bounds__(128)
    decode_merge2(const float* __restrict__ po, const float* __restrict__ plse, const int32_t* __restrict__ mptr,
                  const MergeEnt* __restrict__ ment, OutT* __restrict__ o, float* __restrict__ lse, int Hq, int Hkv,
                  int G) {
    constexpr int C4 = D / 4;
    __shared__ int s_row[kMergeStage];
    __shared__ float s_lse[kMergeStage];
    __shared__ float s_max[8];
    const int r = blockIdx.x / Hkv, kvh = blockIdx.x % Hkv;
    const int e0 = __ldg(mptr + r), E = __ldg(mptr + r + 1) - e0;
    const bool staged = E * G <= kMergeStage;
    if (staged) {
        for (int idx = threadIdx.x; idx < E * G; idx += blockDim.x) {
            const int e = idx / G, j = idx % G;
            const MergeEnt me = ment[e0 + e];
            const int prow = me.pbase + kvh * me.gstride + j;
            s_row[idx] = prow;
            s_lse[idx] = plse[prow];
        }
        __syncthreads();
        if (threadIdx.x < G) {
            float M = -INFINITY;
            for (int e = 0; e < E; ++e) M = fmaxf(M, s_lse[e * G + threadIdx.x]);
            s_max[threadIdx.x] = M;
        }
        __syncthreads();
    }
    for (int u = threadIdx.x; u < G * C4; u += blockDim.x) {
        const int j = u / C4, c4 = u % C4;
        float M;
        if (staged) {
            M = s_max[j];
        } else {
            M = -INFINITY;
            for (int e = 0; e < E; ++e) {
                const MergeEnt me = ment[e0 + e];
                M = fmaxf(M, plse[me.pbase + kvh * me.gstride + j]);
            }
        }
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
        if (M != -INFINITY) {
            int e = 0;
            if (staged) {
                for (; e + 4 <= E; e += 4) {
                    float4 vv[4];
                    float w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int idx = (e + k) * G + j;
                        vv[k] = *(reinterpret_cast<const float4*>(po + (int64_t)s_row[idx] * D) + c4);
                        w[k] = exp2f((s_lse[idx] - M) * kLog2e);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        acc.x += w[k] * vv[k].x;
                        acc.y += w[k] * vv[k].y;
                        acc.z += w[k] * vv[k].z;
                        acc.w += w[k] * vv[k].w;
                        L += w[k];
                    }
                }
            }
            for (; e < E; ++e) {
                int prow;
                float l;
                if (staged) {
                    prow = s_row[e * G + j];
                    l = s_lse[e * G + j];
                } else {
                    const MergeEnt me = ment[e0 + e];
                    prow = me.pbase + kvh * me.gstride + j;
                    l = plse[prow];
                }
                const float w = exp2f((l - M) * kLog2e);
                const float4 vv = *(reinterpret_cast<const float4*>(po + (int64_t)prow * D) + c4);
                acc.x += w * vv.x;
                acc.y += w * vv.y;
                acc.z += w * vv.z;
                acc.w += w * vv.w;
                L += w;
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const int64_t orow = (int64_t)r * Hq + kvh * G + j;
        OutT* dst = o + orow * D + c4 * 4;
        if constexpr (sizeof(OutT) == 2) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(dst) = pk;
        } else {
            *reinterpret_cast<float4*>(dst) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
        if (c4 == 0) lse[orow] = L > 0.f ? M + logf(L) : -INFINITY;
    }
}

}  // namespace

template <int D>
int launch_decode_narrow(const DecItem* items, int n_items, const void* q, const void* kp, const void* vp,
                         const int32_t* r2t, int64_t ld, const int32_t* seq_lens, const int32_t* members, float* po,
                         float* plse, uint32_t* err, int Hq, int Hkv, int G, int64_t num_slots, float scale_log2,
                         cudaStream_t s) {
    if (n_items <= 0) return 0;
    decode_narrow_bf16<D><<<(n_items + 3) / 4, 128, 0, s>>>(
        static_cast<const bf16*>(q), static_cast<const bf16*>(kp), static_cast<const bf16*>(vp), r2t, ld, seq_lens,
        items, n_items, members, po, plse, err, Hq, Hkv, G, num_slots, scale_log2);
    return (int)cudaGetLastError();
}

template <int D>
int launch_decode_merge(bool bf16_out, const float* po, const float* plse, const int32_t* mptr, const MergeEnt* ment,
                        void* o, float* lse, int B, int Hq, int Hkv, int G, cudaStream_t s) {
    if (B <= 0) return 0;
    if (bf16_out)
        decode_merge2<bf16, D><<<B * Hkv, 128, 0, s>>>(po, plse, mptr, ment, static_cast<bf16*>(o), lse, Hq, Hkv, G);
    else
        decode_merge2<float, D><<<B * Hkv, 128, 0, s>>>(po, plse, mptr, ment, static_cast<float*>(o), lse, Hq, Hkv, G);
    return (int)cudaGetLastError();
}

template int launch_decode_narrow<64>(const DecItem*, int, const void*, const void*, const void*, const int32_t*,
                                      int64_t, const int32_t*, const int32_t*, float*, float*, uint32_t*, int, int,
                                      int, int64_t, float, cudaStream_t);
template int launch_decode_narrow<128>(const DecItem*, int, const void*, const void*, const void*, const int32_t*,
                                       int64_t, const int32_t*, const int32_t*, float*, float*, uint32_t*, int, int,
                                       int, int64_t, float, cudaStream_t);
template int launch_decode_merge<64>(bool, const float*, const float*, const int32_t*, const MergeEnt*, void*, float*,
                                     int, int, int, int, cudaStream_t);
template int launch_decode_merge<128>(bool, const float*, const float*, const int32_t*, const MergeEnt*, void*,
                                      float*, int, int, int, int, cudaStream_t);

}  // namespace sgl
