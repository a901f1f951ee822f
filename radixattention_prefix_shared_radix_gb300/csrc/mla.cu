// MLA grouped decode: attention in the 576-dim latent space (CS349D
// lecture-16 notes, SGLang case study: §4 "More engineering", DeepSeek's
// MLA with the decompression matrices absorbed into the query and output
// projections, run by a grouped decode kernel; §5.1 "DP attention": one
// stored row per token, a 512-dim latent plus a 64-dim position part, read
// by every query head).
//
// One CTA (16 warps) per work item of mla_plan.cpp: 64 query rows (member
// request x query head of one head group) against one chunk of a prefix
// segment, in blocks of 32 positions.  A pool row serves as key (all 576
// elements) and, its first 512, as value, so a block's rows are copied into
// shared memory once (16-byte cp.async, three stages, slots looked up three
// blocks ahead by warp 0) and read by both products.  Warps form 4 row
// groups x 4: in S = Q K^T warp (g, w) computes rows 16g.. against positions
// 8w.. over all 576 elements; the four warps of a row group exchange their
// row maxima and then write P (bf16) into a shared tile; in O += P V warp
// (g, w) owns output columns 128w .. 128w + 127 of the group's rows (64
// fp32 accumulators per thread).  Online softmax in base 2 with the scale
// folded in; every block the running max of a row moves to the block max
// when larger and O and the partial sums are rescaled.  Tensor work runs on
// mma.sync m16n8k16 (bf16 in, fp32 accumulate); ldmatrix reads XOR-swizzled
// rows (16-byte chunk c of row r at chunk (c & ~7) | ((c ^ r) & 7)).
// Each item writes normalised partial rows (O fp32, LSE natural log) that
// the log-sum-exp merge (merge.cuh) combines per (request, head group).
#include <cuda_runtime.h>

#include "common.h"
#include "device_common.cuh"
#include "merge.cuh"
#include "mla_tile.cuh"

namespace sgl {
namespace {

using namespace sgldev;

constexpr int kDC = 576;           // stored row: latent + position part
constexpr int kDV = 512;           // output: the latent
constexpr int kBN = 32;            // positions per block
constexpr int kRT = 64;            // query rows per item
constexpr int kStages = 3;         // copy stages
constexpr int kSlotRing = 4;       // slot lists of blocks (one more than the stages)
constexpr int kThreads = 512;      // 16 warps: 4 row groups x 4
constexpr int kRowB = kDC * 2;     // bytes per stored row (bf16)
constexpr int kCPR = kDC / 8;      // 16-byte chunks per row
constexpr int kSPP = kBN + 8;      // pitch of a partial-score row (fp32; the padding spreads the banks)

struct MlaLayout {
    static constexpr int OFF_Q = 0;                                  // [64][576] bf16
    static constexpr int OFF_KV = OFF_Q + kRT * kRowB;               // [stages][32][576] bf16
    static constexpr int OFF_P = OFF_KV + kStages * kBN * kRowB;     // [64][32] bf16
    static constexpr int OFF_SLOT = OFF_P + kRT * kBN * 2;           // [ring][32] int32
    static constexpr int OFF_MX = OFF_SLOT + kSlotRing * kBN * 4;    // [4 groups][4 warps][16] fp32
    static constexpr int OFF_LS = OFF_MX + 16 * 16 * 4;              // the same, for the row sums
    static constexpr int OFF_MEM = OFF_LS + 16 * 16 * 4;             // the item's member requests (at most 4)
    static constexpr int OFF_SP = OFF_MEM + 16;                      // small items: [4 groups][16][kSPP] fp32 partial S
    static constexpr int END = OFF_SP + 4 * 16 * kSPP * 4;
    static constexpr int TOTAL = END + 128;                          // + alignment slack
    static_assert(TOTAL <= 232448, "shared memory per CTA");
};

struct MlaArgs {
    const bf16* q;            // [B, Hq, 576]
    const bf16* kv;           // [num_slots, 576]
    const int32_t* r2t;       // [B, ld]
    int64_t ld;
    const int32_t* seq_lens;  // [B]
    const DecItem* items;
    const int32_t* members;
    float* po;                // partial rows [rows, 512]
    float* plse;              // [rows]
    uint32_t* err;
    int Hq, Gp;
    int64_t num_slots;
    float scale_log2;         // sm_scale * log2(e)
    int n_tile;               // CTAs 0 .. n_tile - 1 run the tcgen05 tile pairs (mla_tile.cuh)
};

// 16-byte chunk c of row r of a [rows][576] bf16 tile
__device__ __forceinline__ uint32_t rswz(int r, int c) {
    return (uint32_t)(r * kRowB + (((c & ~7) | ((c ^ r) & 7)) << 4));
}
// 16-byte chunk c (0..3) of row r of the [64][32] bf16 P tile
__device__ __forceinline__ uint32_t pswz(int r, int c) {
    return (uint32_t)(r * (kBN * 2) + ((c ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__global__ void __launch_bounds__(kThreads, 1) mla_decode_kernel(const __grid_constant__ MlaArgs a,
                                                                 const __grid_constant__ CUtensorMap tmap,
                                                                 const __grid_constant__ CUtensorMap tmq) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if ((int)blockIdx.x < a.n_tile) {
        // a tile pair's output half on the tensor cores
        uint8_t* sm1 = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
        const mlat::TileArgs ta{a.q, a.r2t, a.ld, a.seq_lens, a.items, a.members, a.po, a.plse, a.err,
                                a.Hq, a.Gp, a.num_slots, a.scale_log2};
        mlat::mla_tile_run(ta, &tmap, &tmq, (int)blockIdx.x >> 1, (int)blockIdx.x & 1, sm1, (int)threadIdx.x);
        return;
    }
    uint8_t* sm = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const uint32_t sQ = smem_u32(sm + MlaLayout::OFF_Q), sKV = smem_u32(sm + MlaLayout::OFF_KV);
    const uint32_t sP = smem_u32(sm + MlaLayout::OFF_P);
    int* slots = reinterpret_cast<int*>(sm + MlaLayout::OFF_SLOT);
    float* mxs = reinterpret_cast<float*>(sm + MlaLayout::OFF_MX);
    float* lss = reinterpret_cast<float*>(sm + MlaLayout::OFF_LS);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = warp >> 2, wq = warp & 3, g = lane >> 2, t = lane & 3;
    // the work item is a plan table (uploaded from the host, never written by
    // a kernel): its load overlaps the previous kernel's tail; everything the
    // previous kernel wrote is visible after the dependency wait
    const DecItem it = a.items[blockIdx.x];
    grid_dep_wait();
    grid_dep_launch();
    const int len = __ldg(a.seq_lens + it.rep_row);
    int e = it.kv_end;
    if (e > len) {
        if (tid == 0) atomicOr(a.err, 2u);
        e = len;
    }
    const int b = it.kv_begin;
    const int nb = e > b ? (e - b + kBN - 1) / kBN : 0;
    const int R = it.n_mem * a.Gp;
    const int32_t* trow = a.r2t + (int64_t)it.rep_row * a.ld;

    // slots of block j (warp 0): the raw lookup is issued one block before
    // it is checked and stored (-1 past the range or outside the pool,
    // flagged), so the load never stalls warp 0's share of the math
    auto fetch = [&](int j) -> int {
        const int p = b + j * kBN + lane;
        return (warp == 0 && j < nb && p < e) ? __ldg(trow + p) : -1;
    };
    auto store = [&](int j, int sl) {
        if (warp == 0 && j < nb) {
            if (b + j * kBN + lane < e && (sl < 0 || sl >= a.num_slots)) atomicOr(a.err, 1u);
            slots[(j % kSlotRing) * kBN + lane] = (sl < 0 || sl >= a.num_slots) ? -1 : sl;
        }
    };
    // block j's rows into stage j % kStages (zeros for missing rows); one group
    auto copy = [&](int j) {
        if (j < nb) {
            const uint32_t st = sKV + (uint32_t)((j % kStages) * kBN * kRowB);
            const int* sl = slots + (j % kSlotRing) * kBN;
            for (int i = tid; i < kBN * kCPR; i += kThreads) {
                const int r = i / kCPR, c = i - r * kCPR;
                const int s = sl[r];
                cp_async16(st + rswz(r, c), a.kv + (int64_t)(s < 0 ? 0 : s) * kDC + c * 8, s >= 0);
            }
        }
        cp_async_commit();
    };

    // the first blocks' slot lookups and the item's members (at most 4: the
    // rows' requests) all in flight together, then staged in shared memory
    const int f0 = fetch(0), f1 = fetch(1), f2 = fetch(2);
    int* mems = reinterpret_cast<int*>(sm + MlaLayout::OFF_MEM);
    if (tid < kRT / 16 && tid < it.n_mem) mems[tid] = __ldg(a.members + it.mem_begin + tid);
    store(0, f0);
    store(1, f1);
    store(2, f2);
    int pend = fetch(3);   // block 3's raw slot, stored in the first iteration
    __syncthreads();
    // the item's query rows (zeros past R; a small item reads 16), with block 0's copies
    const int q_rows = R <= 16 ? 16 : kRT;
    for (int i = tid; i < q_rows * kCPR; i += kThreads) {
        const int r = i / kCPR, c = i - r * kCPR;
        const bool ok = r < R;
        const int mem = ok ? mems[r / a.Gp] : 0;
        const int head = it.kvh * a.Gp + (ok ? r % a.Gp : 0);
        cp_async16(sQ + rswz(r, c), a.q + ((int64_t)mem * a.Hq + head) * kDC + c * 8, ok);
    }
    copy(0);
    copy(1);

    if (R <= 16) {
        // ---- an item of at most 16 query rows (a request's own suffix x
        // its heads): every warp takes part in each block.  Row group rg
        // computes S over k-steps 9 rg .. 9 rg + 8 (a quarter of the 576
        // elements) for positions 8 wq .. 8 wq + 7; the four partial scores
        // meet in shared memory and every group sums them in the same order,
        // so all groups hold the same scores and run the same softmax; group
        // 0 writes P, and warp w = 4 rg + wq accumulates output columns
        // 32 w .. 32 w + 31.
        float* sps = reinterpret_cast<float*>(sm + MlaLayout::OFF_SP);
        float o4[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) o4[n][0] = o4[n][1] = o4[n][2] = o4[n][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows g and g + 8
        const int bar_id = 1 + rg;
        for (int j = 0; j < nb; ++j) {
            store(j + 3, pend);
            pend = fetch(j + 4);
            copy(j + 2);
            cp_async_wait<2>();   // block j has landed
            __syncthreads();
            const uint32_t st = sKV + (uint32_t)((j % kStages) * kBN * kRowB);
            {
                constexpr int NQ = kDC / 16 / 4;   // k-steps per row group
                const int k0 = NQ * rg;
                float sp[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t qa[2][4], kb[2][2];
                auto load_s = [&](int ks, int buf) {
                    ldsm_x4(sQ + rswz(lane & 15, 2 * ks + (lane >> 4)), qa[buf][0], qa[buf][1], qa[buf][2],
                            qa[buf][3]);
                    ldsm_x2(st + rswz(8 * wq + (lane & 7), 2 * ks + ((lane >> 3) & 1)), kb[buf][0], kb[buf][1]);
                };
                load_s(k0, 0);
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    if (i + 1 < NQ) load_s(k0 + i + 1, (i + 1) & 1);
                    mma16816(sp, qa[i & 1], kb[i & 1][0], kb[i & 1][1]);
                }
                float* d0 = sps + (rg * 16 + g) * kSPP + 8 * wq + 2 * t;
                *reinterpret_cast<float2*>(d0) = make_float2(sp[0], sp[1]);
                *reinterpret_cast<float2*>(d0 + 8 * kSPP) = make_float2(sp[2], sp[3]);
            }
            __syncthreads();
            float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float* d0 = sps + (k * 16 + g) * kSPP + 8 * wq + 2 * t;
                const float2 ra = *reinterpret_cast<const float2*>(d0);
                const float2 rb = *reinterpret_cast<const float2*>(d0 + 8 * kSPP);
                sum[0] += ra.x;
                sum[1] += ra.y;
                sum[2] += rb.x;
                sum[3] += rb.y;
            }
            const int pos = b + j * kBN + 8 * wq + 2 * t;
            const bool v0 = pos < e, v1 = pos + 1 < e;
            const float x00 = v0 ? sum[0] * a.scale_log2 : -INFINITY;
            const float x01 = v1 ? sum[1] * a.scale_log2 : -INFINITY;
            const float x10 = v0 ? sum[2] * a.scale_log2 : -INFINITY;
            const float x11 = v1 ? sum[3] * a.scale_log2 : -INFINITY;
            float bm0 = fmaxf(x00, x01), bm1 = fmaxf(x10, x11);
            bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 1));
            bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 2));
            bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 1));
            bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 2));
            if (t == 0) {
                mxs[(rg * 4 + wq) * 16 + g] = bm0;
                mxs[(rg * 4 + wq) * 16 + g + 8] = bm1;
            }
            named_bar(bar_id, 128);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                bm0 = fmaxf(bm0, mxs[(rg * 4 + w) * 16 + g]);
                bm1 = fmaxf(bm1, mxs[(rg * 4 + w) * 16 + g + 8]);
            }
            const float n0 = fmaxf(m0, bm0), n1 = fmaxf(m1, bm1);
            const float al0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - n0);
            const float al1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - n1);
            if (n0 > m0 || n1 > m1) {
                l0 *= al0;
                l1 *= al1;
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    o4[n][0] *= al0;
                    o4[n][1] *= al0;
                    o4[n][2] *= al1;
                    o4[n][3] *= al1;
                }
            }
            m0 = n0;
            m1 = n1;
            const float u0 = m0 == -INFINITY ? 0.f : m0, u1 = m1 == -INFINITY ? 0.f : m1;
            const float p00 = exp2f(x00 - u0), p01 = exp2f(x01 - u0), p10 = exp2f(x10 - u1), p11 = exp2f(x11 - u1);
            l0 += p00 + p01;
            l1 += p10 + p11;
            if (rg == 0) {
                asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sP + pswz(g, wq) + 4 * t), "r"(pack_bf16(p00, p01))
                             : "memory");
                asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sP + pswz(g + 8, wq) + 4 * t),
                             "r"(pack_bf16(p10, p11))
                             : "memory");
            }
            __syncthreads();   // P of all 32 positions, for every warp
            {
                uint32_t pa[2][4];
                ldsm_x4(sP + pswz(lane & 15, lane >> 4), pa[0][0], pa[0][1], pa[0][2], pa[0][3]);
                ldsm_x4(sP + pswz(lane & 15, 2 + (lane >> 4)), pa[1][0], pa[1][1], pa[1][2], pa[1][3]);
#pragma unroll
                for (int np = 0; np < 2; ++np) {
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        uint32_t vb[4];
                        ldsm_x4_t(st + rswz(16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8, 4 * warp + 2 * np + (lane >> 4)),
                                  vb[0], vb[1], vb[2], vb[3]);
                        mma16816(o4[2 * np], pa[ks], vb[0], vb[1]);
                        mma16816(o4[2 * np + 1], pa[ks], vb[2], vb[3]);
                    }
                }
            }
            __syncthreads();   // stage j % kStages, P and the partial scores are free again
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
        // row sums over the quad and the group's four warps (every group
        // holds the same sums), then this warp's 32 columns of the rows
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        if (t == 0) {
            lss[(rg * 4 + wq) * 16 + g] = l0;
            lss[(rg * 4 + wq) * 16 + g + 8] = l1;
        }
        named_bar(bar_id, 128);
        float L0 = 0.f, L1 = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            L0 += lss[(rg * 4 + w) * 16 + g];
            L1 += lss[(rg * 4 + w) * 16 + g + 8];
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int row = g + 8 * hh;
            if (row >= R) continue;
            const float L = hh ? L1 : L0, m = hh ? m1 : m0;
            const float inv = L > 0.f ? 1.f / L : 0.f;
            float* dst = a.po + ((int64_t)it.partial_base + row) * kDV + 32 * warp + 2 * t;
#pragma unroll
            for (int n = 0; n < 4; ++n)
                *reinterpret_cast<float2*>(dst + 8 * n) = make_float2(o4[n][2 * hh] * inv, o4[n][2 * hh + 1] * inv);
            if (warp == 0 && t == 0)
                a.plse[(int64_t)it.partial_base + row] = L > 0.f ? (m + log2f(L)) * kLn2 : -INFINITY;
        }
        return;
    }

    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows g and g + 8 of the group
    const int r0 = 16 * rg;                                        // first row of the group
    const bool active = r0 < R;                                    // the group has rows
    const int bar_id = 1 + rg;                                     // named barrier of the group

    for (int j = 0; j < nb; ++j) {
        store(j + 3, pend);
        pend = fetch(j + 4);
        copy(j + 2);
        cp_async_wait<2>();   // groups of blocks <= j + 2 committed: block j has landed
        __syncthreads();
        const uint32_t st = sKV + (uint32_t)((j % kStages) * kBN * kRowB);
        // ---- S for rows r0.., positions 8 wq.. (two accumulators).  The
        // fragments of k-step ks + 2 are loaded before the MMA of ks (the
        // loads and MMAs are volatile asm, kept in source order), so an MMA
        // never waits on the load just before it.
        float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
        if (active) {
            constexpr int NK = kDC / 16;
            uint32_t qa[3][4], kb[3][2];
            auto load_s = [&](int ks, int buf) {
                ldsm_x4(sQ + rswz(r0 + (lane & 15), 2 * ks + (lane >> 4)), qa[buf][0], qa[buf][1], qa[buf][2],
                        qa[buf][3]);
                ldsm_x2(st + rswz(8 * wq + (lane & 7), 2 * ks + ((lane >> 3) & 1)), kb[buf][0], kb[buf][1]);
            };
            load_s(0, 0);
            load_s(1, 1);
#pragma unroll
            for (int ks = 0; ks < NK; ++ks) {
                if (ks + 2 < NK) load_s(ks + 2, (ks + 2) % 3);
                mma16816((ks & 1) ? s2 : s, qa[ks % 3], kb[ks % 3][0], kb[ks % 3][1]);
            }
        }
        const int pos = b + j * kBN + 8 * wq + 2 * t;
        const bool v0 = pos < e, v1 = pos + 1 < e;
        const float x00 = v0 ? (s[0] + s2[0]) * a.scale_log2 : -INFINITY;
        const float x01 = v1 ? (s[1] + s2[1]) * a.scale_log2 : -INFINITY;
        const float x10 = v0 ? (s[2] + s2[2]) * a.scale_log2 : -INFINITY;
        const float x11 = v1 ? (s[3] + s2[3]) * a.scale_log2 : -INFINITY;
        float bm0 = fmaxf(x00, x01), bm1 = fmaxf(x10, x11);
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 1));
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 2));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 1));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 2));
        if (t == 0) {
            mxs[(rg * 4 + wq) * 16 + g] = bm0;
            mxs[(rg * 4 + wq) * 16 + g + 8] = bm1;
        }
        named_bar(bar_id, 128);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            bm0 = fmaxf(bm0, mxs[(rg * 4 + w) * 16 + g]);
            bm1 = fmaxf(bm1, mxs[(rg * 4 + w) * 16 + g + 8]);
        }
        // running max: rescale O and the sums when it grows
        const float n0 = fmaxf(m0, bm0), n1 = fmaxf(m1, bm1);
        const float al0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - n0);
        const float al1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - n1);
        if (n0 > m0 || n1 > m1) {
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                o[n][0] *= al0;
                o[n][1] *= al0;
                o[n][2] *= al1;
                o[n][3] *= al1;
            }
        }
        m0 = n0;
        m1 = n1;
        const float u0 = m0 == -INFINITY ? 0.f : m0, u1 = m1 == -INFINITY ? 0.f : m1;
        const float p00 = exp2f(x00 - u0), p01 = exp2f(x01 - u0), p10 = exp2f(x10 - u1), p11 = exp2f(x11 - u1);
        l0 += p00 + p01;
        l1 += p10 + p11;
        {
            const int ra = r0 + g, rb = r0 + g + 8;
            asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sP + pswz(ra, wq) + 4 * t), "r"(pack_bf16(p00, p01))
                         : "memory");
            asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sP + pswz(rb, wq) + 4 * t), "r"(pack_bf16(p10, p11))
                         : "memory");
        }
        named_bar(bar_id, 128);
        // ---- O[rows r0.., columns 128 wq..] += P V
        if (active) {
            // 16 steps (k-step ks, column pair np): V fragments one step ahead
            uint32_t pa[2][4], vb[2][4];
            ldsm_x4(sP + pswz(r0 + (lane & 15), lane >> 4), pa[0][0], pa[0][1], pa[0][2], pa[0][3]);
            ldsm_x4(sP + pswz(r0 + (lane & 15), 2 + (lane >> 4)), pa[1][0], pa[1][1], pa[1][2], pa[1][3]);
            auto load_v = [&](int step, int buf) {
                const int ks = step >> 3, np = step & 7;
                ldsm_x4_t(st + rswz(16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8, 16 * wq + 2 * np + (lane >> 4)),
                          vb[buf][0], vb[buf][1], vb[buf][2], vb[buf][3]);
            };
            load_v(0, 0);
#pragma unroll
            for (int step = 0; step < 2 * 8; ++step) {
                if (step + 1 < 16) load_v(step + 1, (step + 1) & 1);
                const int ks = step >> 3, np = step & 7, bf = step & 1;
                mma16816(o[2 * np], pa[ks], vb[bf][0], vb[bf][1]);
                mma16816(o[2 * np + 1], pa[ks], vb[bf][2], vb[bf][3]);
            }
        }
        __syncthreads();   // stage j % kStages and P are free again
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");

    // ---- row sums over the quad and the group's four warps, then the rows
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (t == 0) {
        lss[(rg * 4 + wq) * 16 + g] = l0;
        lss[(rg * 4 + wq) * 16 + g + 8] = l1;
    }
    named_bar(bar_id, 128);
    float L0 = 0.f, L1 = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        L0 += lss[(rg * 4 + w) * 16 + g];
        L1 += lss[(rg * 4 + w) * 16 + g + 8];
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int row = r0 + g + 8 * hh;
        if (row >= R) continue;
        const float L = hh ? L1 : L0, m = hh ? m1 : m0;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        float* dst = a.po + ((int64_t)it.partial_base + row) * kDV + 128 * wq + 2 * t;
#pragma unroll
        for (int n = 0; n < 16; ++n)
            *reinterpret_cast<float2*>(dst + 8 * n) = make_float2(o[n][2 * hh] * inv, o[n][2 * hh + 1] * inv);
        if (wq == 0 && t == 0) a.plse[(int64_t)it.partial_base + row] = L > 0.f ? (m + log2f(L)) * kLn2 : -INFINITY;
    }
}

}  // namespace
}  // namespace sgl

extern "C" int sgl_mla_decode_attn(const void* q, const void* kv_pool, const int32_t* req_to_token, int64_t ld,
                                   const int32_t* seq_lens, const sgl_plan* plan, void* o, float* lse,
                                   void* workspace, size_t ws_bytes, sgl_stream_t stream) {
    using namespace sgl;
    if (!plan || plan->kind != 1) return SGL_ERR_INVALID_ARG;
    const sgl_attn_params& p = plan->params;
    if (p.batch > 0 && (!q || !o || !lse || !seq_lens)) return SGL_ERR_INVALID_ARG;
    if (plan->n_items > 0 && (!kv_pool || !req_to_token || ld < plan->max_pos)) return SGL_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) || ws_bytes < plan->workspace_bytes)
        return SGL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_pool) | reinterpret_cast<uintptr_t>(o)) % 16)
        return SGL_ERR_INVALID_ARG;
    auto* ws = static_cast<unsigned char*>(workspace);
    auto s = reinterpret_cast<cudaStream_t>(stream);
    constexpr int kSmem = MlaLayout::TOTAL > mlat::Lay::TOTAL ? MlaLayout::TOTAL : mlat::Lay::TOTAL;
    static const cudaError_t attr =
        cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (attr != cudaSuccess) {
        set_cuda_error((int)attr);
        return SGL_ERR_CUDA;
    }
    MlaArgs a{};
    a.q = static_cast<const bf16*>(q);
    a.kv = static_cast<const bf16*>(kv_pool);
    a.r2t = req_to_token;
    a.ld = ld;
    a.seq_lens = seq_lens;
    a.items = reinterpret_cast<const DecItem*>(ws + plan->off_items);
    a.members = reinterpret_cast<const int32_t*>(ws + plan->off_members);
    a.po = reinterpret_cast<float*>(ws + plan->off_po);
    a.plse = reinterpret_cast<float*>(ws + plan->off_plse);
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.Hq = p.num_qo_heads;
    a.Gp = plan->G;
    a.num_slots = p.num_slots;
    a.scale_log2 = p.sm_scale * kLog2e;
    a.n_tile = plan->n_wide;
    // the tiles' TMA views of the pool, [num_slots, 576] in single rows, and
    // of q, [B * Hq, 576] in boxes of 16 rows (left zero, and unused,
    // without tiles)
    CUtensorMap tmap{}, tmq{};
    if (plan->n_wide > 0) {
        int te = tc::encode_rows_map(kv_pool, p.num_slots, kDC, &tmap);
        if (!te) te = tc::encode_rows_map(q, (int64_t)p.batch * p.num_qo_heads, kDC, &tmq, 16);
        if (te) {
            set_cuda_error(te);
            return SGL_ERR_CUDA;
        }
    }
    // both launches are programmatic dependents of the kernel before them
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cudaError_t e = cudaSuccess;
    if (plan->n_items > 0) {
        cfg.gridDim = dim3((unsigned)plan->n_items);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem;
        e = cudaLaunchKernelEx(&cfg, mla_decode_kernel, a, tmap, tmq);
        if (e != cudaSuccess) {
            set_cuda_error((int)e);
            return SGL_ERR_CUDA;
        }
    }
    if (p.batch == 0) return SGL_OK;
    MergeArgs m{a.po, a.plse, reinterpret_cast<const int32_t*>(ws + plan->off_mptr),
                reinterpret_cast<const int32_t*>(ws + plan->off_ment), o, lse, a.Hq, p.num_kv_heads, plan->G};
    const int n_pairs = p.batch * p.num_kv_heads;
    cfg.gridDim = dim3((unsigned)merge_blocks<kDV>(n_pairs, plan->G));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, decode_merge_kernel<bf16, kDV>, m, n_pairs);
    if (e != cudaSuccess) {
        set_cuda_error((int)e);
        return SGL_ERR_CUDA;
    }
    return SGL_OK;
}
