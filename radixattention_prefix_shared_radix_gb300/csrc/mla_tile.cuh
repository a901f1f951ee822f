// MLA grouped decode on the 5th-generation tensor cores: the shared-prefix
// work of the MLA decode as tcgen05/TMEM tiles (CS349D lecture-16 notes,
// SGLang case study, §4 "More engineering": MLA with the decompression
// matrices absorbed, attention in the 576-dim latent space by a grouped
// decode kernel; §5.1: one stored row per token, read by every query head).
//
// A tile is 128 query rows -- two 64-row work units of the plan (member x
// head of a head group) that read the same chunk of one prefix-group
// segment -- against that chunk, in blocks of 32 positions.  Its output has
// 512 columns (the latent), whose fp32 accumulator for 128 rows alone fills
// all of TMEM, so a tile runs on two CTAs: CTA half h accumulates output
// columns 256 h .. 256 h + 255, and both compute the block's scores.
// Per block j (two score buffers, four K/V stages; the MMA thread issues
// S_0 and S_1, then per block PV_j and S_{j+2}, so the softmax of block
// j + 1 runs while the tensor pipe works on PV_j and S_{j+2}):
//   S_j = Q K_j^T   M 128, N 32, K 576: 36 MMAs, B = the block's rows
//                   (K-major, 128B-swizzled shared memory); A = Q, whose
//                   first 384 elements live in TMEM (24 MMAs with A from
//                   TMEM) and the last 192 in shared memory (12 MMAs);
//   softmax         thread = query row = TMEM lane: the 32 scores, a running
//                   max (O rescaled only when it grows by more than 2^8,
//                   after PV_{j-1} has completed),
//                   P_j = 2^(s - m) as bf16 pairs back into the buffer;
//   O += P_j V_j    M 128, N 256, K 32: A = P from TMEM, B = this half's 256
//                   latent columns of the same shared rows (MN-major).
// Shared memory: four 36 KB stages and Q's last three regions (48 KB).  Q
// arrives by TMA, its first six regions into the last three stages' room;
// the softmax threads move their rows from there into TMEM, after which the
// gathers of blocks 1 .. start (block 0's stage is clear of it).  TMEM:
// O (256 columns), two score buffers (2 x 32), Q (192).
// The stored rows are gathered once per block by TMA tile::gather4 (four
// 128-byte row pieces per copy; the pool viewed as a [slot, 576] tensor with
// 64 x 1 boxes and the 128-byte swizzle) and serve as both K and V.
// Measured on GB300: an M = 128 tcgen05 MMA takes 46 cycles at N = 32,
// 64 at N = 128 and 128 at N = 256 in isolation; here a block's tensor work
// takes ~1.6 us and the block's gather, issued two blocks ahead, lands
// ~4 us after issue, which sets the pace (~2.05 us per block).
// Roles (512 threads): warps 0-3 softmax, warp 4 the MMA thread (and TMEM
// owner), warps 5-15 the gather team (a warp gets one gather4 through about
// every 110 cycles, so a block's 72 copies are spread over eleven warps);
// threads 0-71 issue Q's TMA boxes first.  Before the dependency wait a CTA reads only plan
// tables (its units and their member requests).  Every wait is
// bounded: one that gives up sets bit 2 of the error word and the CTA runs to
// its end without hanging (its results are then garbage, and flagged).
#pragma once

#include <cuda.h>

#include "tc_tile.cuh"

namespace sgl {
namespace mlat {

using namespace sgldev;
using namespace tc;

constexpr int kDC = 576;                  // stored row: latent + position part
constexpr int kDV = 512;                  // output: the latent
constexpr int kBN = 32;                   // positions per block
constexpr int kNS = 4;                    // K/V stages
constexpr int kRows = 128;                // query rows of a tile (two 64-row units)
constexpr int kNReg = kDC / 64;           // 64-element regions of a row: 9
constexpr int kQT = 6;                    // Q regions kept in TMEM (elements 0 .. 383)
constexpr int kQS = kNReg - kQT;          // Q regions kept in shared memory (384 .. 575)
constexpr int kQReg = kRows * 128;        // Q region: 128 rows x 128 bytes
constexpr int kKReg = kBN * 128;          // K/V region of a stage: 32 rows x 128 bytes
constexpr int kStage = kNReg * kKReg;     // 36 KB
constexpr int kNG = 11;                   // gather warps (5 .. 15)
constexpr int kOps = kNReg * (kBN / 4);   // gather4 copies per block: 72
constexpr int kOpw = (kOps + kNG - 1) / kNG;   // per gather warp: 7
constexpr int kOCols = kDV / 2;           // output columns of one CTA: 256
static_assert(kOpw <= 32, "one gather per lane");

struct Lay {
    static constexpr int OFF_KV = 0;                                     // kNS stages
    static constexpr int OFF_Q = OFF_KV + kNS * kStage;                  // 147456: Q regions kQT ..
    static constexpr int OFF_BAR = OFF_Q + kQS * kQReg;                  // 196608
    // Q regions 0 .. kQT - 1 land at the end of the stage area and move to
    // TMEM before any block but the first is gathered
    static constexpr int OFF_QT = OFF_KV + kNS * kStage - kQT * kQReg;   // 49152
    static_assert(OFF_QT >= OFF_KV + kStage, "stage 0 is clear of the Q landing area");
    // barriers: KFULL[kNS], KEMPTY[kNS], SFULL[2], PFULL[2], DONE, QFULL, QMOVED
    static constexpr int KFULL(int s) { return s; }
    static constexpr int KEMPTY(int s) { return kNS + s; }
    static constexpr int SFULL(int b) { return 2 * kNS + b; }
    static constexpr int PFULL(int b) { return 2 * kNS + 2 + b; }
    static constexpr int DONE = 2 * kNS + 4;
    static constexpr int QFULL = DONE + 1;
    static constexpr int QMOVED = DONE + 2;   // Q regions 0 .. kQT - 1 are in TMEM
    static constexpr int kNumBars = DONE + 3;
    static_assert(kNumBars * 8 <= 128, "barrier area");
    // epilogue: this half's O rows (256 fp32 + 16 bytes of pad each) staged
    // in the stage area, which is free once every MMA is done
    static constexpr int OPITCH = kOCols * 4 + 16;
    static_assert(kRows * OPITCH <= kNS * kStage, "the O rows fit the stage area");
    static constexpr int OFF_TMEM = OFF_BAR + 128;
    static constexpr int OFF_MEM = OFF_TMEM + 16;   // the two units' member requests (at most 4 each)
    static constexpr int END = OFF_MEM + 32;
    static constexpr int TOTAL = END + 1024;   // + alignment slack (the 128B swizzle wants 1024-byte alignment)
    static_assert(TOTAL <= 232448, "shared memory per CTA");
};

// TMEM columns: O (this half's 256 columns) first, then the two score
// buffers, then Q's first kQT regions (bf16 pairs, the A operand of the
// first 4 kQT k-steps of S)
constexpr int kTO = 0;
constexpr int kTS = kOCols;
constexpr int kTQ = kTS + 2 * kBN;
static_assert(kTQ + kQT * 32 <= 512, "TMEM columns");

struct TileArgs {
    const bf16* q;            // [B, Hq, 576]
    const int32_t* r2t;       // [B, ld]
    int64_t ld;
    const int32_t* seq_lens;
    const DecItem* items;     // the tile's two units are items 2 t and 2 t + 1
    const int32_t* members;
    float* po;                // partial rows [rows, 512]
    float* plse;
    uint32_t* err;
    int Hq, Gp;
    int64_t num_slots;
    float scale_log2;
};

// 16 TMEM columns of this thread's lane from registers (P: 32 bf16 values)
__device__ __forceinline__ void tst16u(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// One tile half: `t` the tile (items 2 t, 2 t + 1), `h` the output half.
// `sm` is the 1024-aligned shared base, `tid` < 512.
__device__ __forceinline__ void mla_tile_run(const TileArgs& a, const CUtensorMap* tmap, const CUtensorMap* tmq, int t,
                                             int h, uint8_t* sm, int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t sQ = smem_u32(sm + Lay::OFF_Q), sKV = smem_u32(sm + Lay::OFF_KV);
    const uint32_t sQT = smem_u32(sm + Lay::OFF_QT);
    // shared address of Q region reg (the first kQT land in the stage area)
    auto qreg = [&](int reg) { return reg < kQT ? sQT + reg * kQReg : sQ + (reg - kQT) * kQReg; };
    const uint32_t bar0 = smem_u32(sm + Lay::OFF_BAR);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Lay::OFF_TMEM);
    uint32_t* const err = a.err;
    bool timed_out = false;
    auto wait = [&](int b, uint32_t par) {
        if (timed_out) return;
        if (!mbar_wait(bar(b), par)) {
            atomicOr(err, 4u);
            timed_out = true;
        }
    };

    // the tile's units (plan tables) and its chunk
    const DecItem u0 = a.items[2 * t], u1 = a.items[2 * t + 1];
    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(bar(Lay::KFULL(s)), kNG);
            mbar_init(bar(Lay::KEMPTY(s)), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(Lay::SFULL(b)), 1);
            mbar_init(bar(Lay::PFULL(b)), 128);
        }
        mbar_init(bar(Lay::DONE), 1);
        mbar_init(bar(Lay::QFULL), 1);
        mbar_init(bar(Lay::QMOVED), 128);
        mbar_fence_init();
    }
    if (warp == 4) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(tslot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    // before the dependency wait: the units' member requests (plan table)
    // into shared memory and Q's byte count armed
    const int rows0 = u0.n_mem * a.Gp, rows1 = u1.n_mem * a.Gp;
    int* mtab = reinterpret_cast<int*>(sm + Lay::OFF_MEM);
    if (tid < 8) {
        const int u = tid >> 2, k = tid & 3;
        const DecItem& it = u ? u1 : u0;
        mtab[tid] = k < it.n_mem ? __ldg(a.members + it.mem_begin + k) : 0;
    }
    if (tid == 0) mbar_expect_tx(bar(Lay::QFULL), (uint32_t)((rows0 + rows1) / 16 * kNReg * 2048));
    __syncthreads();
    grid_dep_wait();
    grid_dep_launch();
    const int len = __ldg(a.seq_lens + u0.rep_row);   // used once the Q copies are issued

    // Q: 128 rows (unit 0's rows, then unit 1's at 64) x 9 SW128 regions by
    // TMA, 16 rows a box: a member's Gp heads (a multiple of 16) are Gp
    // consecutive rows of q.  Rows past a unit's members are zeroed (their
    // outputs are not written; zeros keep their scores finite).
    {
        const int qunits = 2 * (64 / 16) * kNReg;   // 72 boxes
        if (tid < qunits) {
            const int reg = tid % kNReg, bx = tid / kNReg;   // box: rows 16 bx .. of the tile
            const int r = 16 * bx, u = r >> 6, ri = r & 63;
            if (ri < (u ? rows1 : rows0)) {
                const int mem = mtab[4 * u + ri / a.Gp];
                const int hg = u ? u1.kvh : u0.kvh;
                tma_load_box(qreg(reg) + r * 128, tmq, reg * 64, mem * a.Hq + hg * a.Gp + ri % a.Gp,
                             bar(Lay::QFULL));
            }
        }
        for (int i = tid; i < kRows * 8 * kNReg; i += 512) {   // 16-byte chunks of absent rows
            const int r = i / (8 * kNReg), k = i - r * (8 * kNReg);
            if ((r & 63) >= ((r >> 6) ? rows1 : rows0))
                st_shared_v4(qreg(k >> 3) + r * 128 + (k & 7) * 16, 0u, 0u, 0u, 0u);
        }
    }
    int e = u0.kv_end;
    if (e > len) {
        if (tid == 0) atomicOr(err, 2u);
        e = len;
    }
    const int b = u0.kv_begin;
    const int nb = e > b ? (e - b + kBN - 1) / kBN : 0;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    if (warp >= 5 && warp < 5 + kNG) {
        // ------------------------------------------------------------ gather
        const int g = warp - 5;
        const int o = g * kOpw + lane;
        const int nmine = max(0, min(kOps - g * kOpw, kOpw));
        const bool mine = lane < nmine;
        const int reg = o % kNReg, quad = o / kNReg;
        const int32_t* trow = a.r2t + (int64_t)u0.rep_row * a.ld;
        const uint32_t bytes = (uint32_t)nmine * 512u;
        int issued = 0;
        for (int j = 0; j < nb; ++j) {
            const int st = j % kNS;
            // this lane's four rows (positions past the range re-read the
            // last position: finite data, masked scores)
            int r[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int p = min(b + j * kBN + 4 * quad + k, e - 1);
                int32_t sl = mine ? __ldg(trow + p) : 0;
                if (sl < 0 || sl >= a.num_slots) {
                    if (mine && reg == 0) atomicOr(err, 1u);
                    sl = 0;
                }
                r[k] = sl;
            }
            if (j == 1) wait(Lay::QMOVED, 0);   // stages 1 .. hold Q until it is in TMEM
            wait(Lay::KEMPTY(st), ((j / kNS) & 1) ^ 1);
            if (__any_sync(0xffffffffu, timed_out)) {
                timed_out = true;
                break;
            }
            if (lane == 0) mbar_expect_tx(bar(Lay::KFULL(st)), bytes);
            __syncwarp();
            if (mine)
                tma_gather4(sKV + st * kStage + reg * kKReg + quad * 512, tmap, reg * 64, r[0], r[1], r[2], r[3],
                            bar(Lay::KFULL(st)));
            issued = j + 1;
        }
        // this warp's copies have landed before it leaves (bounded)
        for (int j = max(0, issued - kNS); j < issued; ++j)
            if (!mbar_wait(bar(Lay::KFULL(j % kNS)), (uint32_t)(j / kNS) & 1u)) atomicOr(err, 4u);
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t IS = idesc_bf16(128, kBN, false);
            constexpr uint32_t IO = idesc_bf16(128, kOCols, true);
            // S_j: the first 4 kQT k-steps with A = Q from TMEM, the rest
            // with A = Q's remaining regions in shared memory
            auto mma_s = [&](int j) {
                const uint32_t kb = sKV + (j % kNS) * kStage;
                const uint32_t tS = tbase + kTS + (j & 1) * kBN;
#pragma unroll 4
                for (int ks = 0; ks < 4 * kQT; ++ks)
                    tc_mma_tmem_a(tS, tbase + kTQ + 8 * ks, sdesc(kb + (ks >> 2) * kKReg + (ks & 3) * 32, 16, 1024),
                                  IS, ks > 0);
#pragma unroll 4
                for (int ks = 4 * kQT; ks < kDC / 16; ++ks) {
                    const uint32_t off = (ks & 3) * 32;   // 16 elements within the 64-element region
                    tc_mma(tS, sdesc(sQ + ((ks >> 2) - kQT) * kQReg + off, 16, 1024),
                           sdesc(kb + (ks >> 2) * kKReg + off, 16, 1024), IS, 1u);
                }
                tc_commit(bar(Lay::SFULL(j & 1)));
            };
            // S_0 and S_1; then per block PV_j as soon as P_j is ready (which
            // frees block j's stage for the gather of block j + kNS) and
            // S_{j+2} into block j's score buffer: the softmax of block j + 1
            // runs while the tensor pipe works on PV_j and S_{j+2}
            wait(Lay::QFULL, 0);
            wait(Lay::QMOVED, 0);
            tc_fence_after();
            for (int j = 0; j < 2 && j < nb; ++j) {
                wait(Lay::KFULL(j), 0);
                tc_fence_after();
                mma_s(j);
            }
            for (int j = 0; j < nb; ++j) {
                wait(Lay::PFULL(j & 1), (uint32_t)(j >> 1) & 1u);
                tc_fence_after();
                const uint32_t vb = sKV + (j % kNS) * kStage + 4 * h * kKReg;
                const uint32_t tP = tbase + kTS + (j & 1) * kBN;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    tc_mma_tmem_a(tbase + kTO, tP + kk * 8, sdesc(vb + kk * 2048, kKReg, 1024), IO,
                                  (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar(Lay::KEMPTY(j % kNS)));
                if (j + 2 < nb) {   // into block j's score buffer, read by PV_j (issued before it)
                    wait(Lay::KFULL((j + 2) % kNS), (uint32_t)((j + 2) / kNS) & 1u);
                    tc_fence_after();
                    mma_s(j + 2);
                }
            }
            // every MMA has finished before this thread leaves (bounded)
            tc_commit(bar(Lay::DONE));
            if (!mbar_wait(bar(Lay::DONE), 0)) atomicOr(err, 4u);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ softmax
        const int i = tid;   // row == TMEM lane
        const uint32_t lq = (uint32_t)(warp * 32) << 16;
        const uint32_t tl = tbase + lq;
        const float sc = a.scale_log2;
        float m_used = -INFINITY, l0 = 0.f, l1 = 0.f;
        auto scale_o = [&](float f) {
            float v[32];
#pragma unroll 1
            for (int c = 0; c < kOCols / 32; ++c) {
                tld32(tl + kTO + 32 * c, v);
#pragma unroll
                for (int k = 0; k < 32; ++k) v[k] *= f;
                tst32(tl + kTO + 32 * c, v);
            }
        };
        // this row's Q regions 0 .. kQT - 1 from the landing area into TMEM
        // (a 16-byte chunk = 8 elements = 4 columns of bf16 pairs); the area
        // is then free for the gathers of blocks 1 ..
        wait(Lay::QFULL, 0);
#pragma unroll 1
        for (int reg = 0; reg < kQT; ++reg) {
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t src = sQT + reg * kQReg + i * 128 + ((c ^ (i & 7)) << 4);
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                             : "=r"(w[4 * c]), "=r"(w[4 * c + 1]), "=r"(w[4 * c + 2]), "=r"(w[4 * c + 3])
                             : "r"(src));
            }
            tst32u_nw(tl + kTQ + 32 * reg, w);
        }
        tst_wait();
        tc_fence_before();
        mbar_arrive(bar(Lay::QMOVED));
        for (int j = 0; j < nb; ++j) {
            wait(Lay::SFULL(j & 1), (uint32_t)(j >> 1) & 1u);
            tc_fence_after();
            const uint32_t tS = tl + kTS + (j & 1) * kBN;
            float s[32];
            tld32(tS, s);
            const int pos0 = b + j * kBN;
            if (pos0 + kBN > e) {
#pragma unroll
                for (int k = 0; k < 32; ++k) s[k] = pos0 + k < e ? s[k] : -INFINITY;
            }
            float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
#pragma unroll
                for (int c = 0; c < 4; ++c) mc[c] = fmax3f(mc[c], s[k + 2 * c], s[k + 2 * c + 1]);
            }
            const float mx = fmax3f(mc[0], mc[1], fmaxf(mc[2], mc[3])) * sc;
            const float m_new = fmaxf(m_used, mx);
            const bool need = m_new > m_used + 8.f;   // also true for the first finite max
            const bool resc = need && m_used != -INFINITY;
            if (__any_sync(0xffffffffu, resc)) {
                const float f = resc ? exp2f(m_used - m_new) : 1.f;
                l0 *= f;
                l1 *= f;
                // O holds blocks < j once PV_{j-1} is complete (S_j was
                // issued before it): its stage-release commit says so
                if (j > 0) {
                    wait(Lay::KEMPTY((j - 1) % kNS), (uint32_t)((j - 1) / kNS) & 1u);
                    tc_fence_after();
                    scale_o(f);
                }
            }
            if (need) m_used = m_new;
            const float nmu = m_used == -INFINITY ? 0.f : -m_used;
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                float x0, x1;
                ffma2_sc(x0, x1, s[k], s[k + 1], sc, nmu);
                const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);   // -inf -> 0
                fadd2_acc(l0, l1, p0, p1);
                pk[k / 2] = pack_bf16(p0, p1);
            }
            tst16u(tS, pk);   // P over the scores already read
            tc_fence_before();
            mbar_arrive(bar(Lay::PFULL(j & 1)));
        }
        // epilogue: this half's 256 columns of O / l, once every PV is done
        wait(Lay::DONE, 0);
        tc_fence_after();
        const float l = l0 + l1;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int u = i >> 6, ri = i & 63;
        const bool ok = ri < (u ? rows1 : rows0);
        const int64_t prow = (int64_t)(u ? u1.partial_base : u0.partial_base) + ri;
        // the row through shared memory (padded rows: a warp's 16-byte
        // stores meet no bank twice), out with one bulk copy
        const uint32_t so = sKV + (uint32_t)(i * Lay::OPITCH);
#pragma unroll 1
        for (int c = 0; c < kOCols / 32; c += 2) {
            float v[64];
            if (nb > 0) {
                tld32_nw(tl + kTO + 32 * c, v);
                tld32_nw(tl + kTO + 32 * c + 32, v + 32);
                tld_wait();
            } else {
#pragma unroll
                for (int k = 0; k < 64; ++k) v[k] = 0.f;
            }
#pragma unroll
            for (int k = 0; k < 64; k += 4)
                st_shared_v4(so + (uint32_t)((32 * c + k) * 4), __float_as_uint(v[k] * inv),
                             __float_as_uint(v[k + 1] * inv), __float_as_uint(v[k + 2] * inv),
                             __float_as_uint(v[k + 3] * inv));
        }
        fence_proxy_async_smem();
        if (ok) {
            bulk_s2g(a.po + prow * kDV + kOCols * h, so, (uint32_t)(kOCols * 4));
            bulk_commit();
            if (h == 0) a.plse[prow] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
        }
        bulk_wait_all();   // written before the grid completes
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tbase));
    }
}

}  // namespace mlat
}  // namespace sgl
