// Attention tiles on the 5th-generation tensor cores (tcgen05 + TMEM): NQ
// query tiles of 128 rows against the KV positions [kv_begin, kv_end) of one
// req_to_token row, gathered BN = 128 positions at a time into one K/V
// stream that the query tiles share.  Used by the extend kernel (two query
// tiles per CTA) and by the fused decode kernel (its prefix-group tiles one
// after another).
//
// Roles, by warp of the C::kThreads tile threads:
//   warps 0 .. 4 NQ - 1   softmax: query tile w / 4, thread = query row =
//                         TMEM lane;
//   warp 4 NQ             one thread issues every MMA (the warp owns TMEM);
//   the next NG warps     the gather team: the K and V rows of every block
//                         as TMA tile::gather4 copies (four rows of 128
//                         bytes each, rows of the pool viewed as a 2-D
//                         tensor [slot * Hkv + head, d]) into 128B-swizzled
//                         tiles; extend's Q tiles with 16-byte cp.async.
// Measured on GB300: a warp gets one random-row gather through every ~110
// cycles, whether one lane or many issue them, so the gather rate grows with
// the number of warps that issue; hence a team.
// In single-tile decode configurations Q lives in TMEM (columns after O,
// bf16 pairs, written by the softmax threads from their own rows) and
// S = Q K^T reads A from TMEM, which leaves shared memory to the streaming
// warps; with two query tiles Q is a shared-memory operand.
// The gather team looks up each block's slots in req_to_token one block
// ahead.
// Per 128-position KV block j and query tile q:  S = Q K_j^T (M 128, N 128,
// K d; both operands K-major) into one of NSB TMEM score buffers.  The
// softmax threads read their row in 64-column halves (two TMEM loads in
// flight, one wait), keep a running max m and sum l in base 2 (scores scaled
// by sm_scale*log2 e inside the exponent's FMA), and write P_j = 2^(s - m)
// as bf16 pairs back into the first half of the same TMEM buffer; the MMA
// thread then issues O += P_j V_j with A read from TMEM (M 128, N d, K 128;
// V an MN-major smem operand) and S_{j+NSB} into the freed buffer.  O lives
// in TMEM and is rescaled only when a row's max grows by more than 8 (a
// factor 2^8, harmless in fp32), by the warp that owns the row, which then
// waits for PV_{j-1}; otherwise the softmax never waits for the PV products.
//
// Barrier phases run on across tiles: J counts the blocks and T the tile sets
// this CTA has processed, so a CTA can run any number of tile sets back to
// back (separated by a barrier of the tile threads).  All waits are bounded:
// one that gives up sets bit 2 of the error word and the code runs to its end
// without hanging (its results are then garbage, and flagged).

#pragma once

#include <cuda.h>

#include "device_common.cuh"

namespace sgl {
namespace tc {

using namespace sgldev;

constexpr int kQRegion = 128 * 128;      // SW128 region of a 128-row tile: 128 rows x 128 bytes
constexpr int kTileBar = 1;              // named barrier of the tile threads

// 16-byte chunk c of row r of a bf16 tile kept as 64-column SW128 regions of
// `region` bytes each (the canonical K-major / MN-major 128B-swizzle layout).
__device__ __forceinline__ uint32_t sw128(int r, int c, int region) {
    return (uint32_t)((c >> 3) * region + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16 instruction descriptor: bf16 (or, with f16, f16) A and B, fp32
// D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major, bool f16 = false) {
    return (1u << 4) | (f16 ? 0u : (1u << 7) | (1u << 10)) | (b_mn_major ? (1u << 16) : 0u) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
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
// 32 consecutive TMEM columns of this thread's lane, without waiting for the
// store to complete (tst_wait before the columns are read back or published).
__device__ __forceinline__ void tst32u_nw(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%"
        "18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tst_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tst32u(uint32_t taddr, const uint32_t (&r)[32]) {
    tst32u_nw(taddr, r);
    tst_wait();
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
// 64 consecutive TMEM columns of this thread's lane in one load (measured:
// one x64 load slows concurrent MMAs less than two x32 loads of the same
// columns), without waiting.
__device__ __forceinline__ void tld64_nw(uint32_t taddr, float* v) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,"
        "%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
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
    // extend with the KV write fused in: the new tokens' K/V [n_rows, Hkv, d]
    // (read for the new block instead of the pool) and the pools to write
    // them into; null otherwise
    const bf16* kn;
    const bf16* vn;
    bf16* kw;
    bf16* vw;
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
    // decode with an FP8 (E4M3) pool: per-tensor dequantisation scales (K's
    // goes into the score scale, V's into the normalisation)
    float k_scale, v_scale;
};

// Shared memory of the tile roles (offsets from a 1024-byte aligned base):
// the TMEM base address and a small broadcast area first; everything from
// KEEP on is used only while the tiles run, so a kernel may reuse it once
// its tiles are done: NQ query tiles (extend: 128B-swizzled smem tiles;
// decode: none, Q lives in TMEM), NS K stages and NS V stages of BN
// positions, the barriers and, with FP8 pools, the codes of two blocks' K
// and V rows as copied (BN x D bytes per part) before their conversion into
// the stages.
template <int D, bool DEC, int NQ, int NS, int BN, bool F8 = false>
struct TcLayout {
    static constexpr int OFF_TMEM = 0;                   // TMEM base address
    static constexpr int OFF_INFO = 16;                  // tile description broadcast (16 ints)
    static constexpr int KEEP = 128;
    static constexpr int QTILE = DEC ? 0 : 128 * D * 2;
    static constexpr int KREGION = BN * 128;             // SW128 region: BN rows x 64 columns
    static constexpr int KTILE = BN * D * 2;
    static constexpr int OFF_Q = 1024;
    static constexpr int OFF_K = OFF_Q + NQ * QTILE;
    static constexpr int OFF_V = OFF_K + NS * KTILE;
    static constexpr int OFF_BAR = OFF_V + NS * KTILE;
    static constexpr int OFF_STG = (OFF_BAR + 48 * 8 + 127) / 128 * 128;
    static constexpr int STG = BN * D;
    static constexpr int END = OFF_STG + (F8 ? 4 * STG : 0);
};

// Tile roles and their barriers for NQ query tiles that share one K/V stream
// of NS stages each for K and V, BN positions per block, NSB TMEM score
// buffers per query tile.  Warps 0 .. 4 NQ - 1: softmax (warp w serves query
// tile w / 4, TMEM lanes 32 (w % 4) ..); warp 4 NQ: MMA issue + TMEM owner;
// warps 4 NQ + 1 .. 4 NQ + NG: the gather team.
//
// TMEM columns of query tile q: S buffers at q * 256 + BN b (b < NSB), O at
// q * 256 + NSB * BN; decode's Q after O.  P_j (bf16 pairs) overwrites the
// first BN / 2 columns of its own S buffer.
//
// F8: the pools hold FP8 E4M3 codes.  The gather team copies
// them into a staging area with 16-byte cp.async and stores them, converted
// to f16 (exact), into the same SW128 tiles; Q and P are f16 too, so the MMAs
// are kind::f16 with f16 operands.
template <int D, bool DEC, int NQ, int NS, int NG, int BN, int NSB, bool F8 = false>
struct TcCfg {
    static_assert(NQ == 1 || (NQ == 2 && !DEC), "decode tiles use one query tile (Q lives in TMEM)");
    static_assert(BN == 64 || BN == 128, "KV block of 64 or 128 positions");
    static_assert(NSB == 1 || NSB == 2, "one or two score buffers");
    static_assert(NS >= NSB, "the S lookahead needs as many K stages as score buffers");
    static_assert(NSB * BN + 128 + (DEC ? D / 2 : 0) <= (NQ == 2 ? 256 : 512), "TMEM columns");
    static_assert(NQ == 1 || NSB == 1, "two query tiles alternate on one score buffer each");
    using Lay = TcLayout<D, DEC, NQ, NS, BN, F8>;
    static constexpr int kD = D, kNQ = NQ, kNS = NS, kNG = NG, kBN = BN, kNSB = NSB;
    static constexpr bool kDec = DEC;
    static constexpr bool kF8 = F8;
    static constexpr int kThreads = 32 * (4 * NQ + 1 + NG);
    static constexpr int kMmaWarp = 4 * NQ;
    static constexpr int kOCol = NSB * BN;               // O's column within a query tile's 256
    static constexpr int kQCol = kOCol + 128;            // decode: Q's columns
    // barrier indices
    static constexpr int QFULL = 0;
    static constexpr int KFULL(int s) { return 1 + s; }
    static constexpr int KEMPTY(int s) { return 1 + NS + s; }
    static constexpr int VFULL(int s) { return 1 + 2 * NS + s; }
    static constexpr int VEMPTY(int s) { return 1 + 3 * NS + s; }
    // per query tile: S ready and P ready per score buffer (one barrier per
    // buffer, so the softmax warps can never be two phases ahead of the MMA
    // thread's wait: block j + NSB needs S_{j+NSB}, which is issued only after
    // the MMA thread has consumed block j's P)
    static constexpr int SFULL(int q, int b) { return 1 + 4 * NS + 4 * q + b; }
    static constexpr int PFULL(int q, int b) { return 1 + 4 * NS + 4 * q + 2 + b; }
    // every MMA of the tile set has finished (one phase per tile set, so
    // the waits on it are never ambiguous, unlike a wait on a per-block
    // barrier's last phase when earlier phases may still be pending)
    static constexpr int DONE = 1 + 4 * NS + 4 * NQ;
    static constexpr int kNumBars = DONE + 1;
    static_assert(kNumBars <= 48, "barrier area");
};

// The decode tiles' configuration: one query tile with Q in TMEM, 128-position
// blocks (S MMAs of N = 128), two score buffers so that the softmax of block
// j + 1 overlaps PV_j and S_{j+2}, a gather team of ten warps (every warp of
// the decode CTA has a tile role: a block's 128 gathers of 512 bytes take
// a warp ~110 cycles each to issue, so the block's issue time falls with
// the team's size), and three K/V stages: with the S lookahead a K stage is
// free only once S of the block two earlier has run, and the third stage
// gives the gather of K_{j+2} a whole block more (two with FP8 pools, whose
// staging area takes the room).
template <int D, bool F8 = false>
using DecCfg = TcCfg<D, true, 1, F8 ? 2 : 3, 10, 128, 2, F8>;

struct TileInfo {
    int kv_row, kv_begin, kv_end, kvh;
    int rows[2];   // query rows of each query tile (0: the tile is absent)
    int i6[2];     // extend: first q row of the tile; decode: first member index
    int i7[2];     // extend: causal limit of the tile's row 0; decode: first partial row
    int new_pos;   // fused KV write: first position read from the new K/V (else INT_MAX)
    int new_row;   // fused KV write: the new K/V row of position new_pos
};

struct TcState {
    uint32_t J;        // KV blocks processed by this CTA so far
    uint32_t T;        // tiles processed by this CTA so far
    bool timed_out;
};

// Every barrier of the tile roles invalidated (before their memory is
// reused for something else).
template <class C>
__device__ __forceinline__ void tc_inval_barriers(uint32_t bar0) {
    for (int i = 0; i < C::kNumBars; ++i)
        asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(bar0 + 8u * (uint32_t)i) : "memory");
}

template <class C>
__device__ __forceinline__ void tc_init_barriers(uint32_t bar0) {
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    // Q writers: the softmax threads (decode) or the gather team's lanes (extend)
    mbar_init(bar(C::QFULL), C::kDec ? 128 : 32 * C::kNG);
    // FULL: one arrival per gather warp (an expect_tx whose bytes its TMA
    // gathers complete, or with FP8 pools a plain arrival once its lanes'
    // stores are done); EMPTY: the MMA thread's commit
    for (int s2 = 0; s2 < C::kNS; ++s2) {
        mbar_init(bar(C::KFULL(s2)), C::kNG);
        mbar_init(bar(C::KEMPTY(s2)), 1);
        mbar_init(bar(C::VFULL(s2)), C::kNG);
        mbar_init(bar(C::VEMPTY(s2)), 1);
    }
    for (int q = 0; q < C::kNQ; ++q) {
        for (int b = 0; b < C::kNSB; ++b) {
            mbar_init(bar(C::SFULL(q, b)), 1);
            mbar_init(bar(C::PFULL(q, b)), 128);
        }
    }
    mbar_init(bar(C::DONE), 1);
}

// Run one set of NQ query tiles with the C::kThreads tile threads (tid =
// threadIdx.x < C::kThreads).  `sm` is the 1024-aligned shared base, `tbase`
// the CTA's TMEM columns.  On return the tiles' O / LSE (extend) or partial
// rows (decode) are written by the softmax threads; the caller separates tile
// sets with a barrier of the tile threads.  A query tile with no rows is
// skipped entirely, which keeps the barrier phases consistent only for the
// CTA's last tile set (extend CTAs run one set; decode tiles always have
// rows).
template <class C>
__device__ __forceinline__ void tc_tile_run(const TcArgs& a, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                            const CUtensorMap* tnk, const CUtensorMap* tnv, const TileInfo& ti,
                                            uint8_t* sm, uint32_t tbase, TcState& stt, int tid) {
    using Lay = typename C::Lay;
    constexpr int D = C::kD, NQ = C::kNQ, NS = C::kNS, NG = C::kNG, BN = C::kBN, NSB = C::kNSB;
    constexpr int KR = Lay::KREGION;
    constexpr bool DEC = C::kDec, F8 = C::kF8;
    const uint32_t sQ = smem_u32(sm + Lay::OFF_Q);
    const uint32_t sK = smem_u32(sm + Lay::OFF_K);
    const uint32_t sV = smem_u32(sm + Lay::OFF_V);
    const uint32_t bar0 = smem_u32(sm + Lay::OFF_BAR);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    // argument fields in registers (the asm statements below clobber memory,
    // which would otherwise force a reload through the reference each time)
    const bf16* const a_q = a.q;
    const bf16* const a_kp = a.kp;
    const bf16* const a_vp = a.vp;
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
    const int nb = (kv_end - kv_begin + BN - 1) / BN;
    const uint32_t J0 = stt.J;
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
        const int g = warp - C::kMmaWarp - 1;
        if constexpr (!DEC) {
            // Q: 128 rows per query tile (once, 16-byte cp.async, zero-filled
            // past the tile's rows)
            constexpr int CPR = D / 8;
            constexpr int RPI = 32 / CPR;
            constexpr int QI = 128 / RPI;
            const int sub = lane / CPR, ch = lane % CPR;
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int rq = q ? ti.rows[1] : ti.rows[0], i6q = q ? ti.i6[1] : ti.i6[0];
                for (int t = g; t < QI; t += NG) {
                    const int r = t * RPI + sub;
                    const bool ok = r < rq;
                    const int64_t qr = ((int64_t)i6q + r / a_G) * a_Hq + kvh * a_G + r % a_G;
                    const bf16* src = ok ? a_q + qr * D + ch * 8 : a_q;
                    cp_async16(sQ + q * Lay::QTILE + sw128(r, ch, kQRegion), src, ok);
                }
            }
            if constexpr (F8) {
                // f16 operands against the f16 K tiles: each lane converts
                // the Q chunks it copied, in place, once they have landed
                cp_async_commit();
                cp_async_wait<0>();
                uint32_t qbad = 0u;
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    for (int t = g; t < QI; t += NG) {
                        const uint32_t qa = sQ + q * Lay::QTILE + sw128(t * RPI + sub, ch, kQRegion);
                        uint32_t w[4];
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                     : "r"(qa));
                        st_shared_v4(qa, bf16x2_to_f16x2_chk(w[0], qbad), bf16x2_to_f16x2_chk(w[1], qbad),
                                     bf16x2_to_f16x2_chk(w[2], qbad), bf16x2_to_f16x2_chk(w[3], qbad));
                    }
                }
                if (qbad) atomicOr(a_err, kErrQRange);
                fence_proxy_async_smem();
                mbar_arrive(bar(C::QFULL));
            } else {
                cp_async_arrive_noinc(bar(C::QFULL));
            }
        }
        int issued = 0;
        const int32_t* trow = a_r2t + (int64_t)kv_row * a_ld;
        if constexpr (F8) {
            // FP8 pools: lane t of the team copies 16-code pieces t, t + 32 NG,
            // ... of a block's K and V rows (CH pieces per row) with 16-byte
            // cp.async into one of two staging buffers (no registers held
            // while the codes are in flight; two blocks ahead), then, once
            // the stage is free, reads back its own pieces, converts them to
            // f16 (exact) and stores them into the SW128 tile (two 16-byte
            // chunks per piece); the warp then arrives on the stage's FULL
            // barrier.  A block's slots are looked up one block before its
            // copies are issued and checked only then, so no lookup stalls
            // the conversions.  Positions past the range re-read the range's
            // last position.
            constexpr int CH = D / 16;
            constexpr int NIT = BN * CH;
            constexpr int TPT = (NIT + 32 * NG - 1) / (32 * NG);
            const int t0 = g * 32 + lane;
            const uint8_t* const kp8 = reinterpret_cast<const uint8_t*>(a_kp);
            const uint8_t* const vp8 = reinterpret_cast<const uint8_t*>(a_vp);
            const uint32_t stg = smem_u32(sm + Lay::OFF_STG);
            int32_t sl[TPT];   // slots of this lane's pieces of the next block to copy
            auto lookup = [&](int j) {
#pragma unroll
                for (int i = 0; i < TPT; ++i) {
                    const int it = t0 + i * 32 * NG;
                    const int p = min(kv_begin + j * BN + it / CH, kv_end - 1);
                    sl[i] = (it < NIT && j < nb) ? __ldg(trow + p) : 0;
                }
            };
            // two cp.async groups (K, then V) of block j into staging buffer
            // j & 1; empty groups past the range keep the group count even
            auto copy = [&](int j) {
                const uint32_t sb = stg + (uint32_t)(j & 1) * 2u * Lay::STG;
                int32_t rw[TPT];
#pragma unroll
                for (int i = 0; i < TPT; ++i) {
                    const int it = t0 + i * 32 * NG;
                    int32_t s1 = sl[i];
                    if (s1 < 0 || s1 >= a_num_slots) {
                        if (j < nb && it < NIT && it % CH == 0) atomicOr(a_err, 1u);
                        s1 = 0;
                    }
                    rw[i] = s1 * a_Hkv + kvh;
                }
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    if (j < nb) {
#pragma unroll
                        for (int i = 0; i < TPT; ++i) {
                            const int it = t0 + i * 32 * NG;
                            if (it < NIT)
                                cp_async16(sb + part * Lay::STG + it * 16,
                                           (part ? vp8 : kp8) + (int64_t)rw[i] * D + (it % CH) * 16, true);
                        }
                    }
                    cp_async_commit();
                }
            };
            lookup(0);
            copy(0);
            lookup(1);
            copy(1);
            lookup(2);
            for (int j = 0; j < nb; ++j) {
                const uint32_t J = J0 + j;
                const int st = (int)(J % (uint32_t)NS);
                const uint32_t ph = (J / (uint32_t)NS) & 1u;
                const uint32_t sb = stg + (uint32_t)(j & 1) * 2u * Lay::STG;
                bool stop = false;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    // groups so far: ..., K_j, V_j, K_{j+1}, V_{j+1}
                    if (part == 0)
                        cp_async_wait<3>();
                    else
                        cp_async_wait<2>();
                    wait(part ? C::VEMPTY(st) : C::KEMPTY(st), ph ^ 1u);
                    // store nothing into a stage that may be in use (decided
                    // for the whole warp, which meets at __syncwarp below)
                    if (__any_sync(0xffffffffu, stt.timed_out)) {
                        stt.timed_out = true;
                        stop = true;
                        break;
                    }
                    const uint32_t base = (part ? sV : sK) + st * Lay::KTILE;
#pragma unroll
                    for (int i = 0; i < TPT; ++i) {
                        const int it = t0 + i * 32 * NG;
                        if (it < NIT) {
                            const int r = it / CH, c = it % CH;
                            uint32_t w[4];
                            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                         : "r"(sb + part * Lay::STG + it * 16));
                            uint32_t h[8];
                            e4m3x4_to_f16(w[0], h[0], h[1]);
                            e4m3x4_to_f16(w[1], h[2], h[3]);
                            e4m3x4_to_f16(w[2], h[4], h[5]);
                            e4m3x4_to_f16(w[3], h[6], h[7]);
                            st_shared_v4(base + sw128(r, 2 * c, KR), h[0], h[1], h[2], h[3]);
                            st_shared_v4(base + sw128(r, 2 * c + 1, KR), h[4], h[5], h[6], h[7]);
                        }
                    }
                    // the tensor cores (async proxy) read what these generic
                    // stores wrote: each lane fences its own stores, then one
                    // arrival for the warp
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(part ? C::VFULL(st) : C::KFULL(st)));
                }
                if (stop) break;
                // this buffer is free: block j + 2's codes into it
                copy(j + 2);
                lookup(j + 3);
                issued = j + 1;
            }
            // no copy in flight when the tile ends (the staging area is the
            // next tile's, and the streaming warps' rings overlap it)
            asm volatile("cp.async.wait_all;\n" ::: "memory");
        } else {
            // K and V blocks: NOP TMA gathers each (four rows x 128 bytes: rows
            // 4 quad .. 4 quad + 3, columns 64 half ..), OPW of them per team warp
            // (lane l issues op g OPW + l).  Positions past the range re-read the
            // range's last position (finite data, masked scores), so every row is
            // inside the pool.  With the KV write fused, positions from new_pos on
            // come from the new K/V tensor; a quad that straddles new_pos is
            // loaded as four single rows.
            constexpr int H = D / 64;
            constexpr int NOP = BN / 4 * H;
            constexpr int OPW = (NOP + NG - 1) / NG;
            static_assert(OPW <= 32, "one gather per lane");
            const int o = g * OPW + lane;
            const int nmine = max(0, min(NOP - g * OPW, OPW));   // ops of this warp
            const bool mine = lane < nmine;
            const int half = o % H, quad = o / H;
            const uint32_t bytes = (uint32_t)nmine * 512u;
            const int new_pos = ti.new_pos, new_row = ti.new_row;
            int32_t nx[4];
            int npos0 = 0;   // first position of the quad being fetched
            auto fetch = [&](int j) {
                npos0 = kv_begin + j * BN + 4 * quad;
    #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int p = min(npos0 + i, kv_end - 1);
                    nx[i] = (mine && j < nb && p < new_pos) ? __ldg(trow + p) : 0;
                }
            };
            fetch(0);
            for (int j = 0; j < nb; ++j) {
                const uint32_t J = J0 + j;
                const int st = (int)(J % (uint32_t)NS);
                const uint32_t ph = (J / (uint32_t)NS) & 1u;
                const int npos_cur = npos0;
                int r[4];
                int nsrc = 0;   // rows of the quad read from the new K/V
    #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int p = min(npos_cur + i, kv_end - 1);
                    if (p >= new_pos) {
                        r[i] = (new_row + (p - new_pos)) * a_Hkv + kvh;
                        ++nsrc;
                    } else {
                        int32_t sl = nx[i];
                        if (sl < 0 || sl >= a_num_slots) {
                            if (mine && half == 0) atomicOr(a_err, 1u);
                            sl = 0;
                        }
                        r[i] = sl * a_Hkv + kvh;
                    }
                }
                fetch(j + 1);
                // K rows once S_{j-NS} has read the stage, then V rows once
                // PV_{j-NS} has: separate waits, so that K of a block never waits
                // for a PV product (the MMA thread may need that K before it
                // commits the PV that frees the V stage)
    #pragma unroll
                for (int part = 0; part < 2; ++part) {
                    wait(part ? C::VEMPTY(st) : C::KEMPTY(st), ph ^ 1u);
                    // issue nothing into a stage that may be in use (decided
                    // for the whole warp, which meets at __syncwarp below)
                    if (__any_sync(0xffffffffu, stt.timed_out)) {
                        stt.timed_out = true;
                        break;
                    }
                    const int bfull = part ? C::VFULL(st) : C::KFULL(st);
                    if (lane == 0) mbar_expect_tx(bar(bfull), bytes);
                    __syncwarp();
                    if (mine) {
                        const uint32_t dq = (part ? sV : sK) + st * Lay::KTILE + half * KR + quad * 512;
                        if (nsrc == 0) {
                            tma_gather4(dq, part ? tmv : tmk, half * 64, r[0], r[1], r[2], r[3], bar(bfull));
                        } else if (nsrc == 4) {
                            tma_gather4(dq, part ? tnv : tnk, half * 64, r[0], r[1], r[2], r[3], bar(bfull));
                        } else {
    #pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const bool nw = min(npos_cur + i, kv_end - 1) >= new_pos;
                                tma_load_row(dq + 128 * i, nw ? (part ? tnv : tnk) : (part ? tmv : tmk), half * 64, r[i],
                                             bar(bfull));
                            }
                        }
                    }
                }
                if (stt.timed_out) break;
                issued = j + 1;
            }
        }
        if constexpr (!DEC && !F8) {
            // Fused KV write (after the gathers are issued, so that it overlaps the
            // MMAs): this CTA's new tokens (its query tiles' rows / G)
            // for KV head kvh go from the new K/V into their pool slots.  No
            // CTA reads them from the pool in this launch: positions from
            // new_pos on are gathered from the new K/V themselves.
            if (a.kw != nullptr) {
                constexpr int CH = D / 8;   // 16-byte chunks per row
                const int n0 = ti.rows[0] / a_G, n1 = ti.rows[1] / a_G;
                const int items = (n0 + n1) * 2 * CH;
                const int32_t* trw = a_r2t + (int64_t)kv_row * a_ld;
                for (int it = (g * 32 + lane); it < items; it += NG * 32) {
                    const int ch = it % CH, kvsel = (it / CH) & 1, t = it / (2 * CH);
                    const int row = t < n0 ? ti.i6[0] + t : ti.i6[1] + (t - n0);   // new K/V row
                    const int pos = ti.new_pos + (row - ti.new_row);
                    const int32_t sl = __ldg(trw + pos);
                    if (sl < 0 || sl >= a_num_slots) {
                        if (ch == 0) atomicOr(a_err, 1u);
                        continue;
                    }
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>((kvsel ? a.vn : a.kn) +
                                                                         ((int64_t)row * a_Hkv + kvh) * D) + ch);
                    reinterpret_cast<uint4*>((kvsel ? a.vw : a.kw) + ((int64_t)sl * a_Hkv + kvh) * D)[ch] = v;
                }
            }
        }
        // This warp's copies have landed before it leaves the tile (normally
        // long since: the MMA thread consumed them).  A FULL phase needs this
        // warp's arrival, so the last armed phase of each stage is the one to
        // wait for; the waits are bounded.
        for (int j = F8 ? issued : max(0, issued - NS); j < issued; ++j) {
            const uint32_t J = J0 + j;
            const int st = (int)(J % (uint32_t)NS);
            if (!mbar_wait(bar(C::KFULL(st)), (J / (uint32_t)NS) & 1u)) atomicOr(a_err, 4u);
            if (!mbar_wait(bar(C::VFULL(st)), (J / (uint32_t)NS) & 1u)) atomicOr(a_err, 4u);
        }
        if constexpr (!DEC) asm volatile("cp.async.wait_all;\n" ::: "memory");
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t IS = idesc_bf16(128, BN, false, F8);
            constexpr uint32_t IO = idesc_bf16(128, D, true, F8);
            const bool has0 = ti.rows[0] > 0, has1 = NQ > 1 && ti.rows[1] > 0;
            auto has = [&](int q) { return q ? has1 : has0; };
            wait(C::QFULL, stt.T & 1);
            // extend's Q tiles were written by cp.async (generic proxy) and
            // are read by the tensor cores (async proxy)
            if constexpr (!DEC) fence_proxy_async_smem();
            // S of block j for query tile q into its score buffer
            auto mma_s = [&](int q, uint32_t J, uint32_t kb) {
                const uint32_t tS = tbase + 256 * q + (J % NSB) * BN;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * KR + (ks & 3) * 32;
                    if constexpr (DEC) {
                        tc_mma_tmem_a(tS, tbase + C::kQCol + ks * 8, sdesc(kb + koff, 16, 1024), IS, ks > 0);
                    } else {
                        const uint32_t qoff = q * Lay::QTILE + (ks >> 2) * kQRegion + (ks & 3) * 32;
                        tc_mma(tS, sdesc(sQ + qoff, 16, 1024), sdesc(kb + koff, 16, 1024), IS, ks > 0);
                    }
                }
                tc_commit(bar(C::SFULL(q, J % NSB)));
            };
            auto k_ready = [&](uint32_t J) {
                wait(C::KFULL(J % NS), (J / NS) & 1u);
                tc_fence_after();
                return sK + (J % NS) * Lay::KTILE;
            };
            // S lookahead: the first NSB blocks
            for (int j = 0; j < NSB && j < nb; ++j) {
                const uint32_t kb = k_ready(J0 + j);
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    if (has(q)) mma_s(q, J0 + j, kb);
                tc_commit(bar(C::KEMPTY((J0 + j) % NS)));
            }
            for (int j = 0; j < nb; ++j) {
                const uint32_t J = J0 + j;
                const int st = (int)(J % (uint32_t)NS);
                wait(C::VFULL(st), (J / (uint32_t)NS) & 1u);
                const uint32_t vb = sV + st * Lay::KTILE;
                // S_{j+NSB} reuses block j's score buffer: issued right after
                // PV_j (the tensor pipe runs one thread's MMAs in order)
                const bool next = j + NSB < nb;
                uint32_t kb = 0u;   // K of block j + NSB, waited for once, after the first PV
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    if (!has(q)) continue;
                    wait(C::PFULL(q, J % NSB), (J / NSB) & 1u);
                    tc_fence_after();
                    const uint32_t tP = tbase + 256 * q + (J % NSB) * BN;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        tc_mma_tmem_a(tbase + 256 * q + C::kOCol, tP + kk * 8, sdesc(vb + kk * 2048, KR, 1024), IO,
                                      (j > 0 || kk > 0) ? 1u : 0u);
                    // after the block's last PV: the stage's V is free, and O
                    // holds every block up to j (what a softmax warp that
                    // rescales O waits for; one commit serves both, and a
                    // commit costs the tensor pipe tens of cycles)
                    if (q == NQ - 1 || !has(NQ - 1)) tc_commit(bar(C::VEMPTY(st)));
                    if (next) {
                        if (!kb) kb = k_ready(J + NSB);
                        mma_s(q, J + NSB, kb);
                    }
                }
                if (!has0 && !has1) tc_commit(bar(C::VEMPTY(st)));   // (no PV at all)
                if (next) tc_commit(bar(C::KEMPTY((J + NSB) % NS)));
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
        const uint32_t tlO = tl + C::kOCol;
        const int lim = DEC ? 0x7fffffff : i7 + i / a_G;
        const float sc = F8 ? a_scale * a.k_scale : a_scale;
        float m_used = -INFINITY, l0 = 0.f, l1 = 0.f;   // l = l0 + l1 (packed pair sums)
        if constexpr (DEC) {
            // this row's query (member request i / G, head kvh * G + i % G) into TMEM
            const uint32_t tlQ = tbase + C::kQCol + lq;
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
                if constexpr (F8) {   // f16 operands against the f16 K tiles
                    uint32_t qbad = 0u;
#pragma unroll
                    for (int k = 0; k < 32; ++k) w[k] = bf16x2_to_f16x2_chk(w[k], qbad);
                    if (qbad) atomicOr(a_err, kErrQRange);
                }
                tst32u(tlQ + 32 * c, w);
            }
            tc_fence_before();
            mbar_arrive(bar(C::QFULL));
        }
        // O (rows of this warp) times f, in TMEM
        auto scale_o = [&](float f) {
            float v[32];
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                tld32(tlO + 32 * c, v);
#pragma unroll
                for (int k = 0; k < 32; ++k) v[k] *= f;
                tst32(tlO + 32 * c, v);
            }
        };
        if (rows > 0) {
            for (int j = 0; j < nb; ++j) {
                const uint32_t J = J0 + j;
                const int b = (int)(J % NSB);
                wait(C::SFULL(q, b), (J / NSB) & 1u);
                tc_fence_after();
                // With one score buffer, S_j was issued after PV_{j-1}: O is
                // final for blocks < j.  With two, a warp that rescales waits
                // for PV_{j-1} first, on block j-1's V-stage EMPTY barrier
                // (committed after the block's last PV; that stage's next
                // phase needs PV_{j-1+NS}, hence this warp's P_{j-1+NS}, so
                // the phase waited for is never ambiguous).
                bool o_ready = NSB == 1 || j == 0;
                const uint32_t tS = tl + b * BN;
                // the block in 64-column halves: max, then 2^(s sc - m) as bf16
                // pairs into the block's first BN / 2 columns
#pragma unroll 1
                for (int h = 0; h < BN / 64; ++h) {
                    const int pos0 = kv_begin + j * BN + 64 * h;
                    const bool full_blk = pos0 + 63 < kv_end && pos0 + 63 <= lim;
                    float srow[64];
                    tld64_nw(tS + 64 * h, srow);
                    tld_wait();
                    // max on the raw scores (the scale is positive), scaled
                    // once; four independent chains of 3-input max
                    if (!full_blk) {
#pragma unroll
                        for (int k = 0; k < 64; ++k) {
                            const int pos = pos0 + k;
                            srow[k] = (pos < kv_end && pos <= lim) ? srow[k] : -INFINITY;
                        }
                    }
                    float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int k = 0; k < 64; k += 8) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) mc[c] = fmax3f(mc[c], srow[k + 2 * c], srow[k + 2 * c + 1]);
                    }
                    const float mx = fmax3f(mc[0], mc[1], fmaxf(mc[2], mc[3])) * sc;
                    const float m_new = fmaxf(m_used, mx);
                    const bool need = m_new > m_used + 8.f;   // also true for the first finite max
                    const bool resc = need && m_used != -INFINITY;
                    if (__any_sync(0xffffffffu, resc)) {
                        const float f = resc ? exp2f(m_used - m_new) : 1.f;
                        l0 *= f;
                        l1 *= f;
                        // O holds blocks < j at the old max
                        if (j > 0) {
                            if (!o_ready) {
                                wait(C::VEMPTY((J - 1) % NS), ((J - 1) / NS) & 1u);
                                tc_fence_after();
                                o_ready = true;
                            }
                            scale_o(f);
                        }
                        // this block's earlier halves are at the old max too
                        if (h > 0) tst_wait();   // their P stores have landed
                        for (int h2 = 0; h2 < h; ++h2) {
                            uint32_t w[32];
                            tld32_nw(tS + 32 * h2, reinterpret_cast<float*>(w));
                            tld_wait();
#pragma unroll
                            for (int k = 0; k < 32; ++k) {
                                if constexpr (F8) {
                                    const __half2 v2 = *reinterpret_cast<const __half2*>(&w[k]);
                                    w[k] = pack_f16(__low2float(v2) * f, __high2float(v2) * f);
                                } else {
                                    const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
                                    w[k] = pack_bf16(__low2float(v2) * f, __high2float(v2) * f);
                                }
                            }
                            tst32u(tS + 32 * h2, w);
                        }
                    }
                    if (need) m_used = m_new;
                    const float nmu = m_used == -INFINITY ? 0.f : -m_used;
                    // p = 2^(s sc - m): one packed FMA per pair, one MUFU op
                    // each, one packed add into the pair sums, one conversion
                    // per pair
                    uint32_t pk[32];
#pragma unroll
                    for (int k = 0; k < 64; k += 2) {
                        float x0, x1;
                        ffma2_sc(x0, x1, srow[k], srow[k + 1], sc, nmu);
                        const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);   // -inf -> 0
                        fadd2_acc(l0, l1, p0, p1);
                        pk[k / 2] = F8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
                    }
                    tst32u_nw(tS + 32 * h, pk);   // P over scores already read
                }
                tst_wait();   // the block's P stores have landed before they are published
                tc_fence_before();
                mbar_arrive(bar(C::PFULL(q, b)));
            }
            // epilogue: O / l, two TMEM loads in flight, once every PV is done
            wait(C::DONE, stt.T & 1);
            tc_fence_after();
            const float l = l0 + l1;
            const float inv = l > 0.f ? (F8 ? a.v_scale : 1.f) / l : 0.f;
            const float lse = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
            // decode: the row goes through shared memory (the K/V stages are
            // idle once every MMA is done; rows padded by 16 bytes, so a
            // warp's 16-byte stores meet no bank twice) and out with one bulk
            // copy, instead of 32 lanes storing into 32 rows at once
            constexpr int OPITCH = D * 4 + 16;
            static_assert(!DEC || 128 * OPITCH <= 2 * NS * Lay::KTILE, "the O rows fit the K and V stages");
            const uint32_t so = sK + (uint32_t)(i * OPITCH);
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
                if constexpr (DEC) {
#pragma unroll
                    for (int k = 0; k < 64; k += 4)
                        st_shared_v4(so + (uint32_t)((32 * c + k) * 4), __float_as_uint(v[k] * inv),
                                     __float_as_uint(v[k + 1] * inv), __float_as_uint(v[k + 2] * inv),
                                     __float_as_uint(v[k + 3] * inv));
                } else if (i < rows) {
                    const int64_t orow = ((int64_t)i6 + i / a_G) * a_Hq + kvh * a_G + i % a_G;
                    bf16* dst = a_o + orow * D + 32 * c;
#pragma unroll
                    for (int k = 0; k < 64; k += 8)
                        *reinterpret_cast<uint4*>(dst + k) = make_uint4(
                            pack_bf16(v[k] * inv, v[k + 1] * inv), pack_bf16(v[k + 2] * inv, v[k + 3] * inv),
                            pack_bf16(v[k + 4] * inv, v[k + 5] * inv), pack_bf16(v[k + 6] * inv, v[k + 7] * inv));
                }
            }
            if constexpr (DEC) {
                fence_proxy_async_smem();   // the row's stores, before the async proxy reads them
                if (i < rows) {
                    bulk_s2g(a_po + ((int64_t)i7 + i) * D, so, (uint32_t)(D * 4));
                    bulk_commit();
                    a_plse[(int64_t)i7 + i] = lse;
                }
                bulk_wait_read_all();   // the stages are free again once read
            } else if (i < rows) {
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
// Host: the same view of any [rows, D] bf16 tensor (not cached), with boxes
// of 64 columns x box_rows rows.
int encode_rows_map(const void* base, int64_t rows, int D, CUtensorMap* m, int box_rows = 1);

}  // namespace tc
}  // namespace sgl
