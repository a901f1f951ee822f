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
// and copies each K/V row (head_dim x 2 contiguous bytes of the slot-major
// pool) with 16-byte cp.async into a 128B-swizzled tile, 32/(d/8) rows per
// warp instruction; each lane arrives on the stage's mbarrier when its copies
// land.  K and V have separate 2-stage rings and separate warps, so K_{j+2}
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

#include "device_common.cuh"

namespace sgl {
namespace tc {

using namespace sgldev;

constexpr int kTileThreads = 224;
constexpr int kBN = 64;                  // KV positions per block
constexpr int kQRegion = 128 * 128;      // SW128 region of a 128-row tile: 128 rows x 128 bytes
constexpr int kKRegion = kBN * 128;      // SW128 region of a 64-row tile
constexpr int kTileBar = 1;              // named barrier of the 224 tile threads
constexpr int kSoftmaxBar = 2;           // named barrier of the 128 softmax threads

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

// Shared memory of the tile roles (offsets from a 1024-byte aligned base);
// decode tiles keep Q in TMEM and have no Q tile.
template <int D, bool DEC = false>
struct TcLayout {
    static constexpr int QTILE = DEC ? 0 : 128 * D * 2;
    static constexpr int KTILE = kBN * D * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + QTILE;          // 2 stages
    static constexpr int OFF_V = OFF_K + 2 * KTILE;      // 2 stages
    static constexpr int OFF_BAR = OFF_V + 2 * KTILE;
    static constexpr int OFF_INFO = OFF_BAR + 16 * 8;    // tile description broadcast (8 ints)
    static constexpr int OFF_TMEM = OFF_INFO + 8 * 4;    // TMEM base address
    static constexpr int OFF_MCNT = OFF_TMEM + 4;        // merge list length
    // merge list (128 ints) of a finished decode tile: the K ring is idle then
    static constexpr int OFF_MLIST = OFF_K;
    static constexpr int END = OFF_MCNT + 4;
};

// barrier indices
constexpr int B_QFULL = 0;
constexpr int B_KFULL = 1;     // + stage
constexpr int B_KEMPTY = 3;    // + stage
constexpr int B_VFULL = 5;     // + stage
constexpr int B_VEMPTY = 7;    // + stage
constexpr int B_SFULL = 9;     // + buffer
constexpr int B_PFULL = 11;
constexpr int B_OFULL = 12;
constexpr int kNumBars = 13;

struct TileInfo {
    int kv_row, kv_begin, kv_end, kvh, rows;
    int i6;   // extend: first q row of the tile; decode: first member index
    int i7;   // extend: causal limit of row 0; decode: first partial row
};

struct TcState {
    uint32_t J;        // KV blocks processed by this CTA so far
    uint32_t T;        // tiles processed by this CTA so far
    bool timed_out;
};

template <int D, bool DEC>
__device__ __forceinline__ void tc_init_barriers(uint32_t bar0) {
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    mbar_init(bar(B_QFULL), DEC ? 128 : 64);   // Q writers: softmax threads (decode) / gather lanes (extend)
    for (int s2 = 0; s2 < 2; ++s2) {
        mbar_init(bar(B_KFULL + s2), 32);
        mbar_init(bar(B_KEMPTY + s2), 1);
        mbar_init(bar(B_VFULL + s2), 32);
        mbar_init(bar(B_VEMPTY + s2), 1);
        mbar_init(bar(B_SFULL + s2), 1);
    }
    mbar_init(bar(B_PFULL), 128);
    mbar_init(bar(B_OFULL), 1);
}

// Run one tile with the 224 tile threads (tid = threadIdx.x < 224).  `sm` is
// the 1024-aligned shared base, `tbase` the CTA's TMEM columns (S buffers at
// columns 0 and 64, O at 128; decode: Q at 256, 512 columns allocated).  On return the tile's O / LSE (extend) or
// partial rows (decode) are written by the softmax threads; the caller
// separates tiles with a barrier of the tile threads.
template <int D, bool DEC>
__device__ __forceinline__ void tc_tile_run(const TcArgs& a, const TileInfo& ti, uint8_t* sm, uint32_t tbase,
                                            TcState& stt, int tid) {
    using Lay = TcLayout<D, DEC>;
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
    const int kv_row = ti.kv_row, kv_begin = ti.kv_begin, kv_end = ti.kv_end, kvh = ti.kvh, rows = ti.rows;
    const int i6 = ti.i6, i7 = ti.i7;
    const int nb = (kv_end - kv_begin + kBN - 1) / kBN;
    const uint32_t J0 = stt.J;
    const uint32_t tO = tbase + 128;
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

    if (warp >= 5) {
        // ------------------------------------------------------------ gather
        constexpr int CPR = D / 8;                 // 16-byte chunks per row
        constexpr int RPI = 32 / CPR;              // rows per warp instruction
        const int gw = warp - 5;                   // 0: K, 1: V
        const int sub = lane / CPR, ch = lane % CPR;
        const int32_t* trow = a_r2t + (int64_t)kv_row * a_ld;
        // slots of block 0 (rows lane, lane + 32) before the Q copies
        auto load_slots = [&](int j, int32_t& s0, int32_t& s1) {
            const int p0 = kv_begin + j * kBN + lane, p1 = p0 + 32;
            s0 = (j < nb && p0 < kv_end) ? __ldg(trow + p0) : -1;
            s1 = (j < nb && p1 < kv_end) ? __ldg(trow + p1) : -1;
        };
        int32_t n0, n1;
        load_slots(0, n0, n1);
        if constexpr (!DEC) {
            // Q: this warp's 64 rows
#pragma unroll
            for (int k = 0; k < 64 / RPI; ++k) {
                const int r = gw * 64 + k * RPI + sub;
                const bool ok = r < rows;
                const int64_t qr = ((int64_t)i6 + r / a_G) * a_Hq + kvh * a_G + r % a_G;
                const bf16* src = ok ? a_q + qr * D + ch * 8 : a_q;
                cp_async16(sQ + sw128(r, ch, kQRegion), src, ok);
            }
            cp_async_arrive_noinc(bar(B_QFULL));
        }
        const bf16* pool = gw ? a_vp : a_kp;
        const int bfull = gw ? B_VFULL : B_KFULL, bempty = gw ? B_VEMPTY : B_KEMPTY;
        const uint32_t ring = gw ? sV : sK;
        for (int j = 0; j < nb; ++j) {
            const uint32_t J = J0 + j;
            const int st = J & 1;
            int32_t s0 = n0, s1 = n1;
            load_slots(j + 1, n0, n1);
            const int p0 = kv_begin + j * kBN + lane;
            if (p0 < kv_end && (s0 < 0 || s0 >= a_num_slots)) {
                atomicOr(a_err, 1u);
                s0 = -1;
            }
            if (p0 + 32 < kv_end && (s1 < 0 || s1 >= a_num_slots)) {
                atomicOr(a_err, 1u);
                s1 = -1;
            }
            const uint32_t dst = ring + st * Lay::KTILE;
            wait(bempty + st, ((J >> 1) & 1) ^ 1);
#pragma unroll
            for (int k = 0; k < 64 / RPI; ++k) {
                const int rl = k * RPI + sub;
                const int32_t sr = __shfl_sync(0xffffffffu, (k * RPI < 32) ? s0 : s1, rl & 31);
                const int64_t off = sr >= 0 ? ((int64_t)sr * a_Hkv + kvh) * D + ch * 8 : 0;
                cp_async16(dst + sw128(rl, ch, kKRegion), pool + off, sr >= 0);
            }
            cp_async_arrive_noinc(bar(bfull + st));
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t IS = idesc_bf16(128, kBN, false);
            constexpr uint32_t IO = idesc_bf16(128, D, true);
            wait(B_QFULL, stt.T & 1);
            auto issue_s = [&](int j) {
                const uint32_t J = J0 + j;
                const int st = J & 1;
                wait(B_KFULL + st, (J >> 1) & 1);
                fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t kb = sK + st * Lay::KTILE;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * kKRegion + (ks & 3) * 32;
                    if constexpr (DEC) {
                        tc_mma_tmem_a(tbase + (J & 1) * 64, tQ + ks * 8, sdesc(kb + koff, 16, 1024), IS, ks > 0);
                    } else {
                        const uint32_t qoff = (ks >> 2) * kQRegion + (ks & 3) * 32;
                        tc_mma(tbase + (J & 1) * 64, sdesc(sQ + qoff, 16, 1024), sdesc(kb + koff, 16, 1024), IS,
                               ks > 0);
                    }
                }
                tc_commit(bar(B_SFULL + (J & 1)));
                tc_commit(bar(B_KEMPTY + st));
            };
            if (nb > 0) issue_s(0);
            if (nb > 1) issue_s(1);
            for (int j = 0; j < nb; ++j) {
                const uint32_t J = J0 + j;
                const int st = J & 1;
                wait(B_PFULL, J & 1);
                wait(B_VFULL + st, (J >> 1) & 1);
                fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t vb = sV + st * Lay::KTILE;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    tc_mma_tmem_a(tO, tbase + (J & 1) * 64 + kk * 8, sdesc(vb + kk * 2048, kKRegion, 1024), IO,
                                  (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar(B_OFULL));
                tc_commit(bar(B_VEMPTY + st));
                if (j + 2 < nb) issue_s(j + 2);   // into the buffer P_j occupies: runs after PV_j
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int i = tid;
        const uint32_t tl = tbase + ((uint32_t)(warp * 32) << 16);
        const uint32_t tlO = tO + ((uint32_t)(warp * 32) << 16);
        const int lim = DEC ? 0x7fffffff : i7 + i / a_G;
        const float sc = a_scale;
        float m_used = -INFINITY, l = 0.f;
        if constexpr (DEC) {
            // this row's query (member request i / G, head kvh * G + i % G) into TMEM
            const uint32_t tlQ = tQ + ((uint32_t)(warp * 32) << 16);
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
            mbar_arrive(bar(B_QFULL));
        }
        for (int j = 0; j < nb; ++j) {
            const uint32_t J = J0 + j;
            const int b = J & 1;
            wait(B_SFULL + b, (J >> 1) & 1);
            tc_fence_after();
            const int pos0 = kv_begin + j * kBN;
            const bool full_blk = pos0 + kBN - 1 < kv_end && pos0 + kBN - 1 <= lim;
            float srow[kBN];
            tld32_nw(tl + b * 64, srow);
            tld32_nw(tl + b * 64 + 32, srow + 32);
            tld_wait();
            // max on the raw scores (the scale is positive), scaled once; the
            // scale is folded into the exponent's FMA below
            float mx = -INFINITY;
            if (full_blk) {
#pragma unroll
                for (int k = 0; k < kBN; ++k) mx = fmaxf(mx, srow[k]);
            } else {
#pragma unroll
                for (int k = 0; k < kBN; ++k) {
                    const int pos = pos0 + k;
                    srow[k] = (pos < kv_end && pos <= lim) ? srow[k] : -INFINITY;
                    mx = fmaxf(mx, srow[k]);
                }
            }
            mx *= sc;
            const float m_new = fmaxf(m_used, mx);
            const bool need = m_new > m_used + 8.f;   // also true for the first finite max
            const float m_old = m_used;
            if (need) {
                if (m_used != -INFINITY) l *= exp2f(m_used - m_new);
                m_used = m_new;
            }
            const float nmu = m_used == -INFINITY ? 0.f : -m_used;
            uint32_t pk[kBN / 2];
#pragma unroll
            for (int k = 0; k < kBN; k += 2) {
                const float p0 = exp2f(fmaf(srow[k], sc, nmu));      // -inf -> 0
                const float p1 = exp2f(fmaf(srow[k + 1], sc, nmu));
                l += p0 + p1;
                pk[k / 2] = pack_bf16(p0, p1);
            }
            tst32u(tl + b * 64, pk);                         // P_j over the consumed scores
            // PV_{j-1} is consumed every block (so the barrier is never two
            // phases ahead of this wait); it is normally long done by now.
            if (j > 0) {
                wait(B_OFULL, (J - 1) & 1);
                tc_fence_after();
            }
            // O holds blocks < j scaled to the old max: rescale before PV_j adds to it
            if (j > 0 && __any_sync(0xffffffffu, need && m_old != -INFINITY)) {
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
            mbar_arrive(bar(B_PFULL));
        }
        // epilogue: O / l, two TMEM loads in flight
        if (nb > 0) {
            wait(B_OFULL, (J0 + nb - 1) & 1);
            tc_fence_after();
        }
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
                        *reinterpret_cast<uint4*>(dst + k) =
                            make_uint4(pack_bf16(v[k] * inv, v[k + 1] * inv), pack_bf16(v[k + 2] * inv, v[k + 3] * inv),
                                       pack_bf16(v[k + 4] * inv, v[k + 5] * inv),
                                       pack_bf16(v[k + 6] * inv, v[k + 7] * inv));
                }
            }
        }
        if (i < rows) {
            if constexpr (DEC)
                a_plse[(int64_t)i7 + i] = lse;
            else
                a_lse[((int64_t)i6 + i / a_G) * a_Hq + kvh * a_G + i % a_G] = lse;
        }
        tc_fence_before();
    }
    stt.J = J0 + (uint32_t)(nb > 0 ? nb : 0);
    stt.T += 1;
}

}  // namespace tc
}  // namespace sgl
