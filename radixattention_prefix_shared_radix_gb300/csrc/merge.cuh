// Log-sum-exp merge of decode partials, one warp per (request, query head)
// and slice of at most 128 columns.
//
// Every decode work item writes, for each of its query rows, the softmax-
// normalised partial O over its KV chunk and that chunk's LSE (natural log).
// A request's result for query head j of KV head h combines the E partial
// rows listed for (request, h): with M = max_e lse_e and w_e = exp(lse_e - M),
//   O = sum_e w_e O_e / sum_e w_e,   LSE = M + log(sum_e w_e),
// which equals attention over the concatenated chunks ("SGLang 深度拆解"
// (chenxutan.com/d/5669.html) §3.2 PagedDecode, split along the KV
// sequence).  Every lane accumulates two or four columns of one query head;
// the entries are taken in batches of 16 whose rows and LSEs are all in
// flight together, with the running maximum rescaling earlier batches
// (online form of the same sum).
// Partials are read with ld.global.cg: they were written by other SMs during
// the same kernel (L1 is not coherent).
#pragma once

#include "device_common.cuh"

namespace sgl {

using sgldev::grid_dep_launch;
using sgldev::grid_dep_wait;
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

// One warp merges one slice of one query head's row: all D columns up to
// 128, 128-column slices of wider rows (the MLA latent: four warps per
// head), so that a lane holds at most four columns and sixteen entries'
// rows are in flight together.
template <int D>
struct MergeShape {
    static constexpr int kCols = D < 128 ? D : 128;   // columns per warp
    static constexpr int kSplit = D / kCols;          // warps per (pair, query head)
    static constexpr int kVPL = kCols / 32;           // columns per lane
    static_assert(kVPL == 2 || kVPL == 4, "columns per lane");
};

// Warps (and 128-thread blocks) of a merge launch over n_pairs pairs of G heads.
template <int D>
inline int merge_blocks(int n_pairs, int G) {
    return (n_pairs * G * MergeShape<D>::kSplit + 3) / 4;
}

// Columns col0 .. col0 + kCols - 1 of head j of pair idx = (request, KV
// head), whose entries are ment[e0 .. e0+E): entry e's row for head j is
// ment[e0 + e] + j.  `first` is ment[e0 + lane] for lane < min(E, 32),
// already loaded by the caller.  Every entry row of a batch of 16 is
// requested before the batch's LSEs are used, so a batch costs one round
// trip.
template <typename OutT, int D>
__device__ __noinline__ void merge_head(const MergeArgs& m, int idx, int j, int col0, int e0, int E, int lane,
                                        int first) {
    constexpr int VPL = MergeShape<D>::kVPL;
    constexpr int U = 16;
    const int r = idx / m.Hkv, h = idx - r * m.Hkv;
    float M = -INFINITY, L = 0.f, acc[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) acc[v] = 0.f;
    for (int b = 0; b < E; b += 32) {
        const int n = min(32, E - b);
        const int prow = lane < n ? (b == 0 ? first : __ldg(m.ment + e0 + b + lane)) + j : 0;
        const float ls = lane < n ? __ldcg(m.plse + prow) : -INFINITY;
        for (int k = 0; k < n; k += U) {
            float x[U][VPL], lu[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ok = k + u < n;
                const int pk = __shfl_sync(0xffffffffu, prow, ok ? k + u : 0);
                const float* src = m.po + (int64_t)pk * D + col0 + lane * VPL;
                if constexpr (VPL == 4) {
                    const float4 t4 = ok ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
                    x[u][0] = t4.x;
                    x[u][1] = t4.y;
                    x[u][2] = t4.z;
                    x[u][3] = t4.w;
                } else {
                    const float2 t2 = ok ? __ldcg(reinterpret_cast<const float2*>(src)) : make_float2(0.f, 0.f);
                    x[u][0] = t2.x;
                    x[u][1] = t2.y;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                lu[u] = __shfl_sync(0xffffffffu, ls, k + u < n ? k + u : 0);
                if (k + u >= n) lu[u] = -INFINITY;
            }
            // online form: the running maximum rescales earlier batches
            float mx = M;
#pragma unroll
            for (int u = 0; u < U; ++u) mx = fmaxf(mx, lu[u]);
            if (mx == -INFINITY) continue;
            const float sc = exp2f((M - mx) * kLog2e);   // 0 while nothing was accumulated
            L *= sc;
#pragma unroll
            for (int v = 0; v < VPL; ++v) acc[v] *= sc;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float w = exp2f((lu[u] - mx) * kLog2e);
                L += w;
#pragma unroll
                for (int v = 0; v < VPL; ++v) acc[v] = fmaf(w, x[u][v], acc[v]);
            }
            M = mx;
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int64_t orow = (int64_t)r * m.Hq + h * m.G + j;
    OutT* dst = static_cast<OutT*>(m.o) + orow * D + col0 + lane * VPL;
    if constexpr (sizeof(OutT) == 2) {
        if constexpr (VPL == 4) {
            uint2 pk;
            pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
            pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2*>(dst) = pk;
        } else {
            *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0] * inv, acc[1] * inv);
        }
    } else {
#pragma unroll
        for (int v = 0; v < VPL; ++v) dst[v] = acc[v] * inv;
    }
    if (lane == 0 && col0 == 0) m.lse[orow] = L > 0.f ? M + logf(L) : -INFINITY;
}

// One warp per (request, KV head, query head of the group, column slice):
// the log-sum-exp merge of its entries, or O = 0 / LSE = -inf when the pair
// has no entries (seq_len 0).  The entry range and the first 32 entry rows
// are plan tables (uploaded from the host before the launch before), so
// they are read while the launch before is still running; only the partial
// rows and LSEs, which it writes, are read after the dependency wait.
template <typename OutT, int D>
__global__ void __launch_bounds__(128, 4) decode_merge_kernel(const MergeArgs m, int n_pairs) {
    constexpr int SPLIT = MergeShape<D>::kSplit, COLS = MergeShape<D>::kCols;
    const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int hw = w / SPLIT, sl = w - hw * SPLIT;
    const int idx = hw / m.G, j = hw - idx * m.G;
    int e0 = 0, E = 0, first = 0;
    if (idx < n_pairs) {
        e0 = __ldg(m.mptr + idx);
        E = __ldg(m.mptr + idx + 1) - e0;
        if (lane < E) first = __ldg(m.ment + e0 + lane);
    }
    grid_dep_wait();     // the partials of the launch before
    grid_dep_launch();
    if (idx >= n_pairs) return;
    if (E == 0) {
        const int r = idx / m.Hkv, h = idx - r * m.Hkv;
        const int64_t orow = (int64_t)r * m.Hq + h * m.G + j;
        OutT* dst = static_cast<OutT*>(m.o) + orow * D + sl * COLS;
        for (int c = lane; c < COLS; c += 32) dst[c] = OutT(0.f);
        if (lane == 0 && sl == 0) m.lse[orow] = -INFINITY;
        return;
    }
    merge_head<OutT, D>(m, idx, j, sl * COLS, e0, E, lane, first);
}

}  // namespace sgl
