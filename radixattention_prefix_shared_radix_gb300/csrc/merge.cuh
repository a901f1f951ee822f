// Log-sum-exp merge of decode partials, one warp per (request, KV head).
//
// Every decode work item writes, for each of its query rows, the softmax-
// normalised partial O over its KV chunk and that chunk's LSE (natural log).
// A request's result for query head j of KV head h combines the E partial
// rows listed for (request, h): with M = max_e lse_e and w_e = exp(lse_e - M),
//   O = sum_e w_e O_e / sum_e w_e,   LSE = M + log(sum_e w_e),
// which equals attention over the concatenated chunks ("SGLang 深度拆解"
// (chenxutan.com/d/5669.html) §3.2 PagedDecode, split along the KV
// sequence).  Every lane accumulates D/32 columns of each head; the entries
// are taken in batches whose LSEs and rows are all in flight together, with
// the running maximum rescaling earlier batches (online form of the same
// sum), so a merge costs about two dependent loads plus one per batch.
// Partials are read with ld.global.cg: they were written by other SMs during
// the same kernel (L1 is not coherent).
#pragma once

#include "device_common.cuh"

namespace sgl {

using sgldev::kLog2e;
using sgldev::pack_bf16;

struct MergeArgs {
    const float* po;       // partial rows [rows, D]
    const float* plse;     // partial LSEs [rows]
    const int32_t* mptr;   // [B*Hkv + 1] entry ranges of (request, KV head)
    const int32_t* ment;   // first partial row of each entry (row of head j = ment + j)
    void* o;               // [B, Hq, D] (OutT)
    float* lse;            // [B, Hq]
    int Hq, Hkv, G;
};

template <typename OutT, int D, int G>
__device__ __noinline__ void merge_warp_g(const MergeArgs& m, int idx, int e0, int E, int lane) {
    constexpr int VPL = D / 32;             // columns per lane
    constexpr int U = 24 / G;               // entries whose loads are in flight together
    const int r = idx / m.Hkv, h = idx - r * m.Hkv;
    float M[G], L[G], acc[G][VPL];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        M[j] = -INFINITY;
        L[j] = 0.f;
#pragma unroll
        for (int v = 0; v < VPL; ++v) acc[j][v] = 0.f;
    }
    // Online over batches of U entries: a batch's LSEs and rows are loaded
    // together; the running maxima rescale what was accumulated before.
    for (int b = 0; b < E; b += 32) {
        const int n = min(32, E - b);
        const int pb = lane < n ? __ldg(m.ment + e0 + b + lane) : 0;
        for (int k = 0; k < n; k += U) {
            float x[U][G][VPL], ls[U][G];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ok = k + u < n;
                const int pk = __shfl_sync(0xffffffffu, pb, ok ? k + u : 0);
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    ls[u][j] = ok ? __ldcg(m.plse + pk + j) : -INFINITY;
                    const float* src = m.po + ((int64_t)pk + j) * D + lane * VPL;
                    if constexpr (VPL == 4) {
                        const float4 t = ok ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
                        x[u][j][0] = t.x;
                        x[u][j][1] = t.y;
                        x[u][j][2] = t.z;
                        x[u][j][3] = t.w;
                    } else {
                        const float2 t = ok ? __ldcg(reinterpret_cast<const float2*>(src)) : make_float2(0.f, 0.f);
                        x[u][j][0] = t.x;
                        x[u][j][1] = t.y;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float mx = M[j];
#pragma unroll
                for (int u = 0; u < U; ++u) mx = fmaxf(mx, ls[u][j]);
                if (mx == -INFINITY) continue;
                const float sc = exp2f((M[j] - mx) * kLog2e);   // 0 while nothing was accumulated
                L[j] *= sc;
#pragma unroll
                for (int v = 0; v < VPL; ++v) acc[j][v] *= sc;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float w = exp2f((ls[u][j] - mx) * kLog2e);
                    L[j] += w;
#pragma unroll
                    for (int v = 0; v < VPL; ++v) acc[j][v] = fmaf(w, x[u][j][v], acc[j][v]);
                }
                M[j] = mx;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const float inv = L[j] > 0.f ? 1.f / L[j] : 0.f;
        const int64_t orow = (int64_t)r * m.Hq + h * G + j;
        OutT* dst = static_cast<OutT*>(m.o) + orow * D + lane * VPL;
        if constexpr (sizeof(OutT) == 2) {
            if constexpr (VPL == 4) {
                uint2 pk;
                pk.x = pack_bf16(acc[j][0] * inv, acc[j][1] * inv);
                pk.y = pack_bf16(acc[j][2] * inv, acc[j][3] * inv);
                *reinterpret_cast<uint2*>(dst) = pk;
            } else {
                *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[j][0] * inv, acc[j][1] * inv);
            }
        } else {
#pragma unroll
            for (int v = 0; v < VPL; ++v) dst[v] = acc[j][v] * inv;
        }
        if (lane == 0) m.lse[orow] = L[j] > 0.f ? M[j] + logf(L[j]) : -INFINITY;
    }
}

// Merge pair idx = (request, KV head) whose entries are ment[e0 .. e0+E).
template <typename OutT, int D>
__device__ __forceinline__ void merge_warp(const MergeArgs& m, int idx, int e0, int E, int lane) {
    switch (m.G) {
        case 1: merge_warp_g<OutT, D, 1>(m, idx, e0, E, lane); break;
        case 2: merge_warp_g<OutT, D, 2>(m, idx, e0, E, lane); break;
        case 4: merge_warp_g<OutT, D, 4>(m, idx, e0, E, lane); break;
        default: merge_warp_g<OutT, D, 8>(m, idx, e0, E, lane); break;
    }
}

// (request, KV head) pairs without any partial (seq_len 0): O = 0, LSE = -inf.
template <typename OutT, int D>
__device__ __forceinline__ void merge_empty(const MergeArgs& m, int idx, int lane) {
    const int r = idx / m.Hkv, h = idx - r * m.Hkv;
    for (int j = 0; j < m.G; ++j) {
        const int64_t orow = (int64_t)r * m.Hq + h * m.G + j;
        OutT* dst = static_cast<OutT*>(m.o) + orow * D;
        for (int c = lane; c < D; c += 32) dst[c] = OutT(0.f);
        if (lane == 0) m.lse[orow] = -INFINITY;
    }
}

// One warp per (request, KV head) pair: the log-sum-exp merge of its
// entries, or O = 0 / LSE = -inf for a pair without entries (seq_len 0).
template <typename OutT, int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const MergeArgs m, int n_pairs) {
    const int idx = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (idx >= n_pairs) return;
    const int e0 = __ldg(m.mptr + idx), E = __ldg(m.mptr + idx + 1) - e0;
    if (E == 0)
        merge_empty<OutT, D>(m, idx, lane);
    else
        merge_warp<OutT, D>(m, idx, e0, E, lane);
}

}  // namespace sgl
