// One attention tile on the 5th-generation tensor cores (tcgen05 + TMEM):
// 128 query rows against the KV positions [kv_begin, kv_end) of one
// req_to_token row, gathered 64 positions at a time.  Used by the extend
// kernel (one tile per CTA) and by the fused decode kernel (the CTA's
// prefix-group tiles one after another).
//
// Roles, by warp of the 224 tile threads:
//   warps 0-3  softmax: thread i owns query row i == TMEM lane i;
//   warp  4    one thread issues every MMA (the warp also owns TMEM);
//   warp  5    (extend) gathers half of the Q rows; then the K block of
//              every step;
//   warp  6    (extend) gathers the other Q rows; then the V block of every
//              step.
// Q is a 128B-swizzled smem tile in extend.  In decode tiles it lives in
// TMEM instead (columns 256..256+d/2, bf16 pairs, written by the softmax
// threads from their own rows) and S = Q K^T reads A from TMEM, which leaves
// 64 KB of shared memory to the tile so the fused decode kernel can give the
// rest to its streaming warps.
// A gather warp looks up the block's slots in req_to_token one block ahead
// and fetches the block's 64 K (or V) rows with one warp instruction of TMA
// gathers: each lane issues a tile::gather4 of four rows x 128 bytes (rows
// of the pool viewed as a 2-D tensor [slot * Hkv + head, d]) into the
// 128B-swizzled tile, and lane 0 arms the stage's mbarrier with the block's
// byte count.  Positions past the end of the range re-read the range's last
// position (finite data; their scores are masked), so no row is ever out of
// bounds.  K and V have separate 2-stage rings and separate warps, so K_{j+2}
// loads as soon as S_j is done whatever V is doing.
// Per 64-position KV block j:  S_j = Q K_j^T (M 128, N 64, K d; both operands
// K-major) into one of two TMEM score buffers.  The softmax threads read their
// row (two TMEM loads in flight, one wait), keep a running max m and sum l in
// base 2 (scores pre-scaled by sm_scale*log2 e), and write P_j = 2^(s - m) as
// bf16 pairs back into the first half of the same TMEM buffer; the MMA thread
// then issues O += P_j V_j with A read from TMEM (M 128, N d, K 64; V an
// MN-major smem operand) and S_{j+2} into the freed buffer.  O lives in TMEM
// and is rescaled only when a row's max grows by more than 8 (a factor 2^8,
// harmless in fp32).
//
// Barrier phases run on across tiles: J counts the blocks and T the tiles
// this CTA has processed, so a CTA can run any number of tiles back to back
// (separated by a barrier of the 224 tile threads).  All waits are bounded:
// one that gives up sets bit 2 of the error word and the code runs to its end
// without hanging (its results are then garbage, and flagged).

#pragma once

#include <cuda.h>

#include "device_common.cuh"

namespace sgl {
namespace tc {

using namespace sgldev;

constexpr int kTileThreads = 224;        // threads of a one-query-tile set (7 warps)
constexpr int kBN = 64;                  // KV positions per block
constexpr int kQRegion = 128 * 128;      // SW128 region of a 128-row tile: 128 rows x 128 bytes
constexpr int kKRegion = kBN * 128;      // SW128 region of a 64-row tile
constexpr int kTileBar = 1;              // named barrier of the 224 tile threads

// 16-byte chunk c of row r of a bf16 tile kept as 64-column SW128 regions of
// `region` bytes each (the canonical K-major / MN-major 128B-swizzle layout).
__device__ __forceinline__ uint32_t sw128(int r, int c, int region) {
    return (uint32_t)((c >> 3) * region + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16 instruction descriptor: bf16 A and B, fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// O += A B with A (M x 16) read from TMEM as packed bf16 pairs.
__device__ __forceinline__ void tc_mma_tmem_a(uint32_t tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                              uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::
            "r"(tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tst32u(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%"
        "18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }

// 32 consecutive TMEM columns of this thread's lane, without waiting: several
// can be in flight before one tld_wait().
__device__ __forceinline__ void tld32_nw(uint32_t taddr, float* v) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
        "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tld32(uint32_t taddr, float (&v)[32]) {
    tld32_nw(taddr, v);
    tld_wait();
}

__device__ __forceinline__ void tst32(uint32_t taddr, const float (&v)[32]) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
    tst32u(taddr, r);
}

struct TcArgs {
    const bf16* q;
    const bf16* kp;
    const bf16* vp;
    const int32_t* r2t;
    int64_t ld;
    // extend
    const int32_t* prefix_lens;
    const int32_t* extend_lens;
    int B;
    int64_t n_rows;
    bf16* o;
    float* lse;
    // decode
    const int32_t* seq_lens;
    const DecItem* items;
    const int32_t* members;
    float* po;
    float* plse;
    uint32_t* err;
    int Hq, Hkv, G;
    int64_t num_slots;
    float scale_log2;
};

// Shared memory of the tile roles (offsets from a 1024-byte aligned base):
// NQ query tiles (extend: 128B-swizzled smem tiles; decode: none, Q lives in
// TMEM), NSK K stages and NSV V stages of 64 positions, the barriers and a
// small broadcast area.
template <int D, bool DEC, int NQ, int NSK, int NSV>
struct TcLayout {
    static constexpr int QTILE = DEC ? 0 : 128 * D * 2;
    static constexpr int KTILE = kBN * D * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NQ * QTILE;
    static constexpr int OFF_V = OFF_K + NSK * KTILE;
    static constexpr int OFF_BAR = OFF_V + NSV * KTILE;
    static constexpr int OFF_INFO = OFF_BAR + 48 * 8;    // tile description broadcast (16 ints)
    static constexpr int OFF_TMEM = OFF_INFO + 16 * 4;   // TMEM base address
    static constexpr int END = OFF_TMEM + 16;
};

// Tile roles and their barriers for NQ query tiles that share one K/V stream
// of NSK + NSV stages.  Warps 0 .. 4 NQ - 1: softmax (warp w serves query
// tile w / 4, TMEM lanes 32 (w % 4) ..); warp 4 NQ: MMA issue + TMEM owner;
// warp 4 NQ + 1: K gathers; warp 4 NQ + 2: V gathers.
template <int D, bool DEC, int NQ, int NSK, int NSV>
struct TcCfg {
    static_assert(NQ == 1 || (NQ == 2 && !DEC), "decode tiles use one query tile (Q lives in TMEM)");
    static_assert(NSK >= 2 && NSV >= 2, "the S lookahead needs two K stages");
    using Lay = TcLayout<D, DEC, NQ, NSK, NSV>;
    static constexpr int kD = D, kNQ = NQ, kNSK = NSK, kNSV = NSV;
    static constexpr bool kDec = DEC;
    static constexpr int kThreads = 32 * (4 * NQ + 3);
    static constexpr int kMmaWarp = 4 * NQ;
    static constexpr int kTmemCols = (DEC || NQ == 2) ? 512 : 256;
    // barrier indices
    static constexpr int QFULL = 0;
    static constexpr int KFULL(int s) { return 1 + s; }
    static constexpr int KEMPTY(int s) { return 1 + NSK + s; }
    static constexpr int VFULL(int s) { return 1 + 2 * NSK + s; }
    static constexpr int VEMPTY(int s) { return 1 + 2 * NSK + NSV + s; }
    // per query tile: S ready and P ready per TMEM score buffer b = block & 1
    // (one barrier per buffer, so the softmax warps can never be two phases
    // ahead of the MMA thread's wait: block j + 2 needs S_{j+2}, which is
    // issued only after the MMA thread has consumed block j's P), O updated
    static constexpr int SFULL(int q, int b) { return 1 + 2 * NSK + 2 * NSV + 5 * q + b; }
    static constexpr int PFULL(int q, int b) { return 1 + 2 * NSK + 2 * NSV + 5 * q + 2 + b; }
    static constexpr int OFULL(int q) { return 1 + 2 * NSK + 2 * NSV + 5 * q + 4; }
    // every MMA of the tile set has finished (one phase per tile set, so
    // the waits on it are never ambiguous, unlike a wait on OFULL's last
    // phase when earlier phases may still be pending)
    static constexpr int DONE = 1 + 2 * NSK + 2 * NSV + 5 * NQ;
    static constexpr int kNumBars = DONE + 1;
    static_assert(kNumBars <= 48, "barrier area");
};

// The decode tiles' configuration (one query tile, Q in TMEM, 2 + 2 stages).
template <int D>
using DecCfg = TcCfg<D, true, 1, 2, 2>;

struct TileInfo {
    int kv_row, kv_begin, kv_end, kvh;
    int rows[2];   // query rows of each query tile (0: the tile is absent)
    int i6[2];     // extend: first q row of the tile; decode: first member index
    int i7[2];     // extend: causal limit of the tile's row 0; decode: first partial row
};

struct TcState {
    uint32_t J;        // KV blocks processed by this CTA so far
    uint32_t T;        // tiles processed by this CTA so far
    bool timed_out;
};

template <class C>
__device__ __forceinline__ void tc_init_barriers(uint32_t bar0) {
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    mbar_init(bar(C::QFULL), C::kDec ? 128 : 64);   // Q writers: softmax threads (decode) / gather lanes (extend)
    // FULL: lane 0's expect_tx (the TMA gathers complete the bytes); EMPTY:
    // the MMA thread's commit
    for (int s2 = 0; s2 < C::kNSK; ++s2) {
        mbar_init(bar(C::KFULL(s2)), 1);
        mbar_init(bar(C::KEMPTY(s2)), 1);
    }
    for (int s2 = 0; s2 < C::kNSV; ++s2) {
        mbar_init(bar(C::VFULL(s2)), 1);
        mbar_init(bar(C::VEMPTY(s2)), 1);
    }
    for (int q = 0; q < C::kNQ; ++q) {
        mbar_init(bar(C::SFULL(q, 0)), 1);
        mbar_init(bar(C::SFULL(q, 1)), 1);
        mbar_init(bar(C::PFULL(q, 0)), 128);
        mbar_init(bar(C::PFULL(q, 1)), 128);
        mbar_init(bar(C::OFULL(q)), 1);
    }
    mbar_init(bar(C::DONE), 1);
}

// Run one set of NQ query tiles with the C::kThreads tile threads (tid =
// threadIdx.x < C::kThreads).  `sm` is the 1024-aligned shared base, `tbase`
// the CTA's TMEM columns: query tile q has its S buffers at columns
// 256 q + {0, 64} and O at 256 q + 128; decode keeps Q at column 256.  On
// return the tiles' O / LSE (extend) or partial rows (decode) are written by
// the softmax threads; the caller separates tile sets with a barrier of the
// tile threads.  A query tile with no rows is skipped entirely, which keeps
// the barrier phases consistent only for the CTA's last tile set (extend
// CTAs run one set; decode tiles always have rows).
template <class C>
__device__ __forceinline__ void tc_tile_run(const TcArgs& a, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                            const TileInfo& ti, uint8_t* sm, uint32_t tbase, TcState& stt, int tid) {
    using Lay = typename C::Lay;
    constexpr int D = C::kD, NQ = C::kNQ, NSK = C::kNSK, NSV = C::kNSV;
    constexpr bool DEC = C::kDec;
    const uint32_t sQ = smem_u32(sm + Lay::OFF_Q);
    const uint32_t sK = smem_u32(sm + Lay::OFF_K);
    const uint32_t sV = smem_u32(sm + Lay::OFF_V);
    const uint32_t bar0 = smem_u32(sm + Lay::OFF_BAR);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    // argument fields in registers (the asm statements below clobber memory,
    // which would otherwise force a reload through the reference each time)
    const bf16* const a_q = a.q;
    const int32_t* const a_r2t = a.r2t;
    const int64_t a_ld = a.ld;
    const int32_t* const a_members = a.members;
    float* const a_po = a.po;
    float* const a_plse = a.plse;
    bf16* const a_o = a.o;
    float* const a_lse = a.lse;
    uint32_t* const a_err = a.err;
    const int a_Hq = a.Hq, a_Hkv = a.Hkv, a_G = a.G;
    const int64_t a_num_slots = a.num_slots;
    const float a_scale = a.scale_log2;
    const int warp = tid >> 5, lane = tid & 31;
    const int kv_row = ti.kv_row, kv_begin = ti.kv_begin, kv_end = ti.kv_end, kvh = ti.kvh;
    const int nb = (kv_end - kv_begin + kBN - 1) / kBN;
    const uint32_t J0 = stt.J;
    const uint32_t tQ = tbase + 256;
    // after one wait has given up, the tile's results are garbage (flagged):
    // later waits return at once so the CTA finishes promptly
    auto wait = [&](int b, uint32_t par) {
        if (stt.timed_out) return;
        if (!mbar_wait(bar(b), par)) {
            atomicOr(a_err, 4u);
            stt.timed_out = true;
        }
    };

    if (warp > C::kMmaWarp) {
        // ------------------------------------------------------------ gather
        const int gw = warp - C::kMmaWarp - 1;     // 0: K, 1: V
        if constexpr (!DEC) {
            // Q: rows 64 gw .. 64 gw + 63 of every query tile (once, 16-byte cp.async)
            constexpr int CPR = D / 8;             // 16-byte chunks per row
            constexpr int RPI = 32 / CPR;          // rows per warp instruction
            const int sub = lane / CPR, ch = lane % CPR;
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
#pragma unroll
                for (int k = 0; k < 64 / RPI; ++k) {
                    const int r = gw * 64 + k * RPI + sub;
                    const bool ok = r < (q ? ti.rows[1] : ti.rows[0]);
                    const int64_t qr = ((int64_t)(q ? ti.i6[1] : ti.i6[0]) + r / a_G) * a_Hq + kvh * a_G + r % a_G;
                    const bf16* src = ok ? a_q + qr * D + ch * 8 : a_q;
                    cp_async16(sQ + q * Lay::QTILE + sw128(r, ch, kQRegion), src, ok);
                }
            }
            cp_async_arrive_noinc(bar(C::QFULL));
        }
        // lane = (half, quad): rows 4 quad .. 4 quad + 3, columns 64 half ..
        constexpr int H = D / 64;                  // 128-byte halves of a row
        constexpr int NS = NSK > NSV ? NSK : NSV;
        const int ns = gw ? NSV : NSK;
        const int quad = lane & 15, half = lane >> 4;
        const int32_t* trow = a_r2t + (int64_t)kv_row * a_ld;
        int32_t nx[4];
        auto fetch = [&](int j) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int p = min(kv_begin + j * kBN + 4 * quad + i, kv_end - 1);
                nx[i] = j < nb ? __ldg(trow + p) : 0;
            }
        };
        fetch(0);
        const CUtensorMap* tm = gw ? tmv : tmk;
        const uint32_t ring = gw ? sV : sK;
        int issued = 0;
        for (int j = 0; j < nb; ++j) {
            const uint32_t J = J0 + j;
            const int st = (int)(J % (uint32_t)ns);
            const uint32_t ph = (J / (uint32_t)ns) & 1u;
            int r[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                int32_t sl = nx[i];
                if (sl < 0 || sl >= a_num_slots) {
                    if (half == 0) atomicOr(a_err, 1u);
                    sl = 0;
                }
                r[i] = sl * a_Hkv + kvh;
            }
            fetch(j + 1);
            wait(gw ? C::VEMPTY(st) : C::KEMPTY(st), ph ^ 1u);
            if (stt.timed_out) break;   // issue nothing into a stage that may be in use
            const int bfull = gw ? C::VFULL(st) : C::KFULL(st);
            if (lane == 0) mbar_expect_tx(bar(bfull), (uint32_t)(kBN * D * 2));
            __syncwarp();
            if (half < H)
                tma_gather4(ring + st * Lay::KTILE + half * kKRegion + quad * 512, tm, half * 64, r[0], r[1], r[2],
                            r[3], bar(bfull));
            issued = j + 1;
        }
        // This warp's copies have landed before it leaves the tile (normally
        // long since: the MMA thread consumed them).  Only this warp arms the
        // FULL barriers, so the last armed phase of each stage is the one to
        // wait for; the waits are bounded.
        for (int j = max(0, issued - ns); j < issued; ++j) {
            const uint32_t J = J0 + j;
            const int st = (int)(J % (uint32_t)ns);
            if (!mbar_wait(bar(gw ? C::VFULL(st) : C::KFULL(st)), (J / (uint32_t)ns) & 1u)) atomicOr(a_err, 4u);
        }
        (void)NS;
        if constexpr (!DEC) asm volatile("cp.async.wait_all;\n" ::: "memory");
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t IS = idesc_bf16(128, kBN, false);
            constexpr uint32_t IO = idesc_bf16(128, D, true);
            const bool has0 = ti.rows[0] > 0, has1 = NQ > 1 && ti.rows[1] > 0;
            auto has = [&](int q) { return q ? has1 : has0; };
            wait(C::QFULL, stt.T & 1);
            // extend's Q tiles were written by cp.async (generic proxy) and
            // are read by the tensor cores (async proxy)
            if constexpr (!DEC) fence_proxy_async_smem();
            auto issue_s = [&](int j) {
                const uint32_t J = J0 + j;
                const int st = (int)(J % (uint32_t)NSK);
                wait(C::KFULL(st), (J / (uint32_t)NSK) & 1u);
                tc_fence_after();
                const uint32_t kb = sK + st * Lay::KTILE;
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    if (!has(q)) continue;
                    const uint32_t tS = tbase + 256 * q + (J & 1) * 64;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t koff = (ks >> 2) * kKRegion + (ks & 3) * 32;
                        if constexpr (DEC) {
                            tc_mma_tmem_a(tS, tQ + ks * 8, sdesc(kb + koff, 16, 1024), IS, ks > 0);
                        } else {
                            const uint32_t qoff = q * Lay::QTILE + (ks >> 2) * kQRegion + (ks & 3) * 32;
                            tc_mma(tS, sdesc(sQ + qoff, 16, 1024), sdesc(kb + koff, 16, 1024), IS, ks > 0);
                        }
                    }
                    tc_commit(bar(C::SFULL(q, J & 1)));
                }
                tc_commit(bar(C::KEMPTY(st)));
            };
            if (nb > 0) issue_s(0);
            if (nb > 1) issue_s(1);
            for (int j = 0; j < nb; ++j) {
                const uint32_t J = J0 + j;
                const int st = (int)(J % (uint32_t)NSV);
                wait(C::VFULL(st), (J / (uint32_t)NSV) & 1u);
                const uint32_t vb = sV + st * Lay::KTILE;
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    if (!has(q)) continue;
                    wait(C::PFULL(q, J & 1), (J >> 1) & 1);
                    tc_fence_after();
                    const uint32_t tP = tbase + 256 * q + (J & 1) * 64;
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        tc_mma_tmem_a(tbase + 256 * q + 128, tP + kk * 8, sdesc(vb + kk * 2048, kKRegion, 1024), IO,
                                      (j > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar(C::OFULL(q)));
                }
                tc_commit(bar(C::VEMPTY(st)));
                if (j + 2 < nb) issue_s(j + 2);   // into the buffers P_j occupies: runs after PV_j
            }
            // every MMA of the tile set has finished before this thread
            // leaves it (the commit covers all earlier MMAs; bounded wait)
            tc_commit(bar(C::DONE));
            if (!mbar_wait(bar(C::DONE), stt.T & 1)) atomicOr(a_err, 4u);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int q = NQ == 1 ? 0 : warp >> 2;     // query tile of this warp
        const int i = tid - 128 * q;               // row within the tile == TMEM lane
        // (selects, not indexing: a run-time index would put ti in local memory)
        const int rows = q ? ti.rows[1] : ti.rows[0], i6 = q ? ti.i6[1] : ti.i6[0], i7 = q ? ti.i7[1] : ti.i7[0];
        const uint32_t lq = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tl = tbase + 256 * q + lq;
        const uint32_t tlO = tl + 128;
        const int lim = DEC ? 0x7fffffff : i7 + i / a_G;
        const float sc = a_scale;
        float m_used = -INFINITY, l0 = 0.f, l1 = 0.f;   // l = l0 + l1 (packed pair sums)
        if constexpr (DEC) {
            // this row's query (member request i / G, head kvh * G + i % G) into TMEM
            const uint32_t tlQ = tQ + lq;
            const bool ok = i < rows;
            const int mem = ok ? __ldg(a_members + i6 + i / a_G) : 0;
            const uint4* src = reinterpret_cast<const uint4*>(a_q + ((int64_t)mem * a_Hq + kvh * a_G + i % a_G) * D);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t w[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 v = ok ? __ldg(src + 8 * c + k) : make_uint4(0, 0, 0, 0);
                    w[4 * k] = v.x;
                    w[4 * k + 1] = v.y;
                    w[4 * k + 2] = v.z;
                    w[4 * k + 3] = v.w;
                }
                tst32u(tlQ + 32 * c, w);
            }
            tc_fence_before();
            mbar_arrive(bar(C::QFULL));
        }
        if (rows > 0) {
            for (int j = 0; j < nb; ++j) {
                const uint32_t J = J0 + j;
                const int b = J & 1;
                wait(C::SFULL(q, b), (J >> 1) & 1);
                tc_fence_after();
                const int pos0 = kv_begin + j * kBN;
                const bool full_blk = pos0 + kBN - 1 < kv_end && pos0 + kBN - 1 <= lim;
                float srow[kBN];
                tld32_nw(tl + b * 64, srow);
                tld32_nw(tl + b * 64 + 32, srow + 32);
                tld_wait();
                // max on the raw scores (the scale is positive), scaled once;
                // the scale is folded into the exponent's FMA below.  Four
                // independent chains of 3-input max keep the dependency chain
                // short.
                if (!full_blk) {
#pragma unroll
                    for (int k = 0; k < kBN; ++k) {
                        const int pos = pos0 + k;
                        srow[k] = (pos < kv_end && pos <= lim) ? srow[k] : -INFINITY;
                    }
                }
                float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int k = 0; k < kBN; k += 8) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) mc[c] = fmax3f(mc[c], srow[k + 2 * c], srow[k + 2 * c + 1]);
                }
                const float mx = fmax3f(mc[0], mc[1], fmaxf(mc[2], mc[3])) * sc;
                const float m_new = fmaxf(m_used, mx);
                const bool need = m_new > m_used + 8.f;   // also true for the first finite max
                const float m_old = m_used;
                if (need) {
                    if (m_used != -INFINITY) {
                        const float f = exp2f(m_used - m_new);
                        l0 *= f;
                        l1 *= f;
                    }
                    m_used = m_new;
                }
                const float nmu = m_used == -INFINITY ? 0.f : -m_used;
                // p = 2^(s sc - m): one packed FMA per pair, one MUFU op each,
                // one packed add into the pair sums, one conversion per pair
                uint32_t pk[kBN / 2];
#pragma unroll
                for (int k = 0; k < kBN; k += 2) {
                    float x0, x1;
                    ffma2_sc(x0, x1, srow[k], srow[k + 1], sc, nmu);
                    const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);   // -inf -> 0
                    fadd2_acc(l0, l1, p0, p1);
                    pk[k / 2] = pack_bf16(p0, p1);
                }
                tst32u(tl + b * 64, pk);                         // P_j over the consumed scores
                // O holds blocks < j scaled to the old max: a warp with a row
                // whose max grew rescales its rows once PV_{j-1} has finished.
                // Other warps do not touch O and go on without waiting: the
                // OFULL barrier cannot run two phases ahead of a waiter (its
                // next phase needs this warp's P_j), so skipped waits are safe.
                if (j > 0 && __any_sync(0xffffffffu, need && m_old != -INFINITY)) {
                    wait(C::OFULL(q), (J - 1) & 1);
                    tc_fence_after();
                    const float al = (need && m_old != -INFINITY) ? exp2f(m_old - m_new) : 1.f;
                    float v[32];
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        tld32(tlO + 32 * c, v);
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] *= al;
                        tst32(tlO + 32 * c, v);
                    }
                }
                tc_fence_before();
                mbar_arrive(bar(C::PFULL(q, b)));
            }
            // epilogue: O / l, two TMEM loads in flight, once every PV is done
            wait(C::DONE, stt.T & 1);
            tc_fence_after();
            const float l = l0 + l1;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const float lse = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
#pragma unroll 1
            for (int c = 0; c < D / 32; c += 2) {
                float v[64];
                if (nb > 0) {
                    tld32_nw(tlO + 32 * c, v);
                    tld32_nw(tlO + 32 * c + 32, v + 32);
                    tld_wait();
                } else {
#pragma unroll
                    for (int k = 0; k < 64; ++k) v[k] = 0.f;
                }
                if (i < rows) {
                    if constexpr (DEC) {
                        float* dst = a_po + ((int64_t)i7 + i) * D + 32 * c;
#pragma unroll
                        for (int k = 0; k < 64; k += 4)
                            *reinterpret_cast<float4*>(dst + k) =
                                make_float4(v[k] * inv, v[k + 1] * inv, v[k + 2] * inv, v[k + 3] * inv);
                    } else {
                        const int64_t orow = ((int64_t)i6 + i / a_G) * a_Hq + kvh * a_G + i % a_G;
                        bf16* dst = a_o + orow * D + 32 * c;
#pragma unroll
                        for (int k = 0; k < 64; k += 8)
                            *reinterpret_cast<uint4*>(dst + k) = make_uint4(
                                pack_bf16(v[k] * inv, v[k + 1] * inv), pack_bf16(v[k + 2] * inv, v[k + 3] * inv),
                                pack_bf16(v[k + 4] * inv, v[k + 5] * inv), pack_bf16(v[k + 6] * inv, v[k + 7] * inv));
                    }
                }
            }
            if (i < rows) {
                if constexpr (DEC)
                    a_plse[(int64_t)i7 + i] = lse;
                else
                    a_lse[((int64_t)i6 + i / a_G) * a_Hq + kvh * a_G + i % a_G] = lse;
            }
        }
        tc_fence_before();
    }
    stt.J = J0 + (uint32_t)(nb > 0 ? nb : 0);
    stt.T += 1;
}

// Host: tensor maps of the K and V pools viewed as 2-D bf16 tensors
// [num_slots * Hkv rows, D columns] with 64 x 1 boxes and the 128-byte
// swizzle, for the tile gathers.  The last maps made on this thread are
// reused while the pools and shape are the same.  Returns a cudaError_t.
int encode_pool_maps(const void* kp, const void* vp, int64_t num_slots, int Hkv, int D, CUtensorMap* mk,
                     CUtensorMap* mv);

}  // namespace tc
}  // namespace sgl
