// Attention over gathered KV on the 5th-generation tensor cores (tcgen05 +
// TMEM), for tiles of 128 query rows against 128-position KV blocks.
//
// Two users:
//   * extend ("SGLang 深度拆解" (chenxutan.com/d/5669.html) §3.2 PagedPrefill;
//     "SGLang 深度解读" section "5. Attention 层"): rows = (new token x query
//     head of one KV head), 128/G new tokens per tile; positions 0..p of the
//     request's req_to_token row, causal inside the new block;
//   * wide decode items: a prefix-group segment shared by many requests; rows
//     = (member request x query head), all reading the same chunk of the
//     segment's representative row once ("SGLang：从前端 DSL 到 SRT 服务运行时",
//     section "用基数树实现前缀复用"); output = normalised partial rows merged
//     later by log-sum-exp.
//
// CTA roles (224 threads; two CTAs share an SM, so two independent tiles keep
// the tensor core and the softmax units busy in turn):
//   warps 0-3  softmax: thread i owns query row i == TMEM lane i;
//   warp  4    allocates TMEM (256 columns); one thread issues every MMA;
//   warps 5-6  gather: slot lookup in req_to_token and 16-byte cp.async of the
//              K and V rows (head_dim x 2 contiguous bytes each in the
//              slot-major pool) into 128B-swizzled tiles, consecutive lanes on
//              consecutive chunks of a row; each thread signals the stage's
//              mbarrier when its copies land.  K and V have separate 2-stage
//              rings: K_{j+2} may load as soon as S_j is done.
// Per 64-position KV block j:  S_j = Q K_j^T (M 128, N 64, K d; both operands
// K-major) into one of two TMEM score buffers.  The softmax threads read their
// row (two TMEM loads in flight, one wait), keep a running max m and sum l in
// base 2 (scores pre-scaled by sm_scale*log2 e), and write P_j = 2^(s - m) as
// bf16 pairs back into the first half of the same TMEM buffer; the MMA thread
// then issues O += P_j V_j with A read from TMEM (M 128, N d, K 64; V an
// MN-major smem operand) and S_{j+2} into the freed buffer.  O lives in TMEM
// and is rescaled only when a row's max grows by more than 8 (a factor 2^8,
// harmless in fp32).  All waits are bounded: one that gives up sets bit 2 of
// the workspace error word and the kernel runs to its end without hanging
// (its results are then garbage, and flagged).

#include "device_common.cuh"

namespace sgl {
namespace {

using namespace sgldev;

constexpr int kTcThreads = 224;
constexpr int kBN = 64;                  // KV positions per block
constexpr int kQRegion = 128 * 128;      // SW128 region of a 128-row tile: 128 rows x 128 bytes
constexpr int kKRegion = kBN * 128;      // SW128 region of a 64-row tile

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

__device__ __forceinline__ void tld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
        "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// Same load without the wait: several can be in flight before one tld_wait().
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

__device__ __forceinline__ void tst32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%"
        "18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
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
    // wide decode items
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

template <int D>
struct TcLayout {
    static constexpr int QTILE = 128 * D * 2;
    static constexpr int KTILE = kBN * D * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + QTILE;          // 2 stages
    static constexpr int OFF_V = OFF_K + 2 * KTILE;      // 2 stages
    static constexpr int OFF_BAR = OFF_V + 2 * KTILE;
    static constexpr int OFF_INFO = OFF_BAR + 16 * 8;
    static constexpr int OFF_TMEM = OFF_INFO + 16 * 4;
    static constexpr int TOTAL = OFF_TMEM + 16 + 1024;   // + alignment slack
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

template <bool DEC>
__device__ void tile_setup(const TcArgs& a, int* info) {
    // info: 0 valid, 1 kv_row, 2 kv_begin, 3 kv_end, 4 kvh, 5 rows, 6 qrow0|mem_begin, 7 lim0|partial_base
    info[0] = 0;
    if constexpr (DEC) {
        const DecItem it = a.items[blockIdx.x];
        int e = it.kv_end;
        const int len = __ldg(a.seq_lens + it.rep_row);
        if (e > len) {
            atomicOr(a.err, 2u);
            e = len;
        }
        info[1] = it.rep_row;
        info[2] = it.kv_begin;
        info[3] = e > it.kv_begin ? e : it.kv_begin;
        info[4] = it.kvh;
        info[5] = it.n_mem * a.G;
        info[6] = it.mem_begin;
        info[7] = it.partial_base;
        info[0] = 1;
    } else {
        const int tq = 128 / a.G;
        int acc_t = 0, acc_q = 0, req = -1, tile0 = 0, qoff = 0;
        for (int r = 0; r < a.B; ++r) {
            const int e = __ldg(a.extend_lens + r);
            const int nt = e > 0 ? (e + tq - 1) / tq : 0;
            if ((int)blockIdx.x < acc_t + nt) {
                req = r;
                tile0 = acc_t;
                qoff = acc_q;
                break;
            }
            acc_t += nt;
            acc_q += e > 0 ? e : 0;
        }
        if (req < 0) return;
        const int pre = __ldg(a.prefix_lens + req), ext = __ldg(a.extend_lens + req);
        const int t0 = ((int)blockIdx.x - tile0) * tq;
        const int ntok = min(tq, ext - t0);
        if (pre < 0 || ntok <= 0 || (int64_t)pre + ext > a.ld || (int64_t)qoff + t0 + ntok > a.n_rows) {
            atomicOr(a.err, 2u);
            return;
        }
        info[1] = req;
        info[2] = 0;
        info[3] = pre + t0 + ntok;
        info[4] = blockIdx.y;
        info[5] = ntok * a.G;
        info[6] = qoff + t0;
        info[7] = pre + t0;
        info[0] = 1;
    }
}

template <int D, bool DEC>
__global__ void __maxnreg__(128) tc_attn_kernel(const TcArgs a) {
    using Lay = TcLayout<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sQ = smem_u32(sm + Lay::OFF_Q);
    const uint32_t sK = smem_u32(sm + Lay::OFF_K);
    const uint32_t sV = smem_u32(sm + Lay::OFF_V);
    const uint32_t bar0 = smem_u32(sm + Lay::OFF_BAR);
    int* info = reinterpret_cast<int*>(sm + Lay::OFF_INFO);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Lay::OFF_TMEM);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) tile_setup<DEC>(a, info);
    __syncthreads();
    if (!info[0]) return;
    const int kv_row = info[1], kv_begin = info[2], kv_end = info[3], kvh = info[4], rows = info[5];
    const int i6 = info[6], i7 = info[7];
    const int nb = (kv_end - kv_begin + kBN - 1) / kBN;

    if (tid == 0) {
        mbar_init(bar(B_QFULL), 64);
        for (int s2 = 0; s2 < 2; ++s2) {
            mbar_init(bar(B_KFULL + s2), 64);
            mbar_init(bar(B_KEMPTY + s2), 1);
            mbar_init(bar(B_VFULL + s2), 64);
            mbar_init(bar(B_VEMPTY + s2), 1);
            mbar_init(bar(B_SFULL + s2), 1);
        }
        mbar_init(bar(B_PFULL), 128);
        mbar_init(bar(B_OFULL), 1);
        mbar_fence_init();
    }
    if (warp == 4) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;\n" ::"r"(smem_u32(tslot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;     // S buffers at columns 0 and 64, O at 128
    const uint32_t tO = tbase + 128;
    bool timed_out = false;
    auto wait = [&](int b, uint32_t par) {
        if (!mbar_wait(bar(b), par)) {
            if (!timed_out) atomicOr(a.err, 4u);
            timed_out = true;
        }
    };

    if (warp >= 5) {
        // ------------------------------------------------------------ gather
        constexpr int CPR = D / 8;                 // 16-byte chunks per row
        constexpr int RPI = 32 / CPR;              // rows per warp instruction
        const int gw = warp - 5;
        const int sub = lane / CPR, ch = lane % CPR;
#pragma unroll 4
        for (int k = 0; k < 64 / RPI; ++k) {       // 64 query rows per gather warp
            const int r = gw * 64 + k * RPI + sub;
            const bool ok = r < rows;
            const bf16* src = a.q;
            if (ok) {
                int64_t qr;
                if constexpr (DEC)
                    qr = (int64_t)__ldg(a.members + i6 + r / a.G) * a.Hq + kvh * a.G + r % a.G;
                else
                    qr = ((int64_t)i6 + r / a.G) * a.Hq + kvh * a.G + r % a.G;
                src = a.q + qr * D + ch * 8;
            }
            cp_async16(sQ + sw128(r, ch, kQRegion), src, ok);
        }
        cp_async_arrive_noinc(bar(B_QFULL));
        const int32_t* trow = a.r2t + (int64_t)kv_row * a.ld;
        const int myrow = gw * 32 + lane;          // this lane looks up the slot of row myrow
        int32_t raw_next = (nb > 0 && kv_begin + myrow < kv_end) ? __ldg(trow + kv_begin + myrow) : -1;
        for (int j = 0; j < nb; ++j) {
            const int st = j & 1;
            const uint32_t par = ((j >> 1) & 1) ^ 1;
            const int pos = kv_begin + j * kBN + myrow;
            int32_t s = raw_next;
            raw_next = (j + 1 < nb && pos + kBN < kv_end) ? __ldg(trow + pos + kBN) : -1;
            bool ok = pos < kv_end;
            if (ok && (s < 0 || s >= a.num_slots)) {
                atomicOr(a.err, 1u);
                ok = false;
            }
            if (!ok) s = -1;
            const uint32_t kd = sK + st * Lay::KTILE, vd = sV + st * Lay::KTILE;
            wait(B_KEMPTY + st, par);
#pragma unroll 4
            for (int k = 0; k < 32 / RPI; ++k) {
                const int rl = k * RPI + sub;
                const int32_t sr = __shfl_sync(0xffffffffu, s, rl);
                const int64_t off = sr >= 0 ? ((int64_t)sr * a.Hkv + kvh) * D + ch * 8 : 0;
                cp_async16(kd + sw128(gw * 32 + rl, ch, kKRegion), a.kp + off, sr >= 0);
            }
            cp_async_arrive_noinc(bar(B_KFULL + st));
            wait(B_VEMPTY + st, par);
#pragma unroll 4
            for (int k = 0; k < 32 / RPI; ++k) {
                const int rl = k * RPI + sub;
                const int32_t sr = __shfl_sync(0xffffffffu, s, rl);
                const int64_t off = sr >= 0 ? ((int64_t)sr * a.Hkv + kvh) * D + ch * 8 : 0;
                cp_async16(vd + sw128(gw * 32 + rl, ch, kKRegion), a.vp + off, sr >= 0);
            }
            cp_async_arrive_noinc(bar(B_VFULL + st));
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t IS = idesc_bf16(128, kBN, false);
            constexpr uint32_t IO = idesc_bf16(128, D, true);
            wait(B_QFULL, 0);
            auto issue_s = [&](int j) {
                const int st = j & 1;
                wait(B_KFULL + st, (j >> 1) & 1);
                fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t kb = sK + st * Lay::KTILE;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t qoff = (ks >> 2) * kQRegion + (ks & 3) * 32;
                    const uint32_t koff = (ks >> 2) * kKRegion + (ks & 3) * 32;
                    tc_mma(tbase + (j & 1) * 64, sdesc(sQ + qoff, 16, 1024), sdesc(kb + koff, 16, 1024), IS, ks > 0);
                }
                tc_commit(bar(B_SFULL + (j & 1)));
                tc_commit(bar(B_KEMPTY + st));
            };
            if (nb > 0) issue_s(0);
            if (nb > 1) issue_s(1);
            for (int j = 0; j < nb; ++j) {
                const int st = j & 1;
                wait(B_PFULL, j & 1);
                wait(B_VFULL + st, (j >> 1) & 1);
                fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t vb = sV + st * Lay::KTILE;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    tc_mma_tmem_a(tO, tbase + (j & 1) * 64 + kk * 8, sdesc(vb + kk * 2048, kKRegion, 1024), IO,
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
        const int lim = DEC ? 0x7fffffff : i7 + i / a.G;
        const float sc = a.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        for (int j = 0; j < nb; ++j) {
            const int b = j & 1;
            wait(B_SFULL + b, (j >> 1) & 1);
            tc_fence_after();
            const int pos0 = kv_begin + j * kBN;
            const bool full_blk = pos0 + kBN - 1 < kv_end && pos0 + kBN - 1 <= lim;
            float srow[kBN];
            tld32_nw(tl + b * 64, srow);
            tld32_nw(tl + b * 64 + 32, srow + 32);
            tld_wait();
            float mx = -INFINITY;
            if (full_blk) {
#pragma unroll
                for (int k = 0; k < kBN; ++k) {
                    srow[k] *= sc;
                    mx = fmaxf(mx, srow[k]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < kBN; ++k) {
                    const int pos = pos0 + k;
                    srow[k] = (pos < kv_end && pos <= lim) ? srow[k] * sc : -INFINITY;
                    mx = fmaxf(mx, srow[k]);
                }
            }
            const float m_new = fmaxf(m_used, mx);
            const bool need = m_new > m_used + 8.f;   // also true for the first finite max
            const float m_old = m_used;
            if (need) {
                if (m_used != -INFINITY) l *= exp2f(m_used - m_new);
                m_used = m_new;
            }
            const float mu = m_used == -INFINITY ? 0.f : m_used;
            uint32_t pk[kBN / 2];
#pragma unroll
            for (int k = 0; k < kBN; k += 2) {
                const float p0 = exp2f(srow[k] - mu);      // -inf -> 0
                const float p1 = exp2f(srow[k + 1] - mu);
                l += p0 + p1;
                pk[k / 2] = pack_bf16(p0, p1);
            }
            tst32u(tl + b * 64, pk);                         // P_j over the consumed scores
            // PV_{j-1} is consumed every block (so the barrier is never two
            // phases ahead of this wait); it is normally long done by now.
            if (j > 0) {
                wait(B_OFULL, (j - 1) & 1);
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
        // epilogue
        if (nb > 0) {
            wait(B_OFULL, (nb - 1) & 1);
            tc_fence_after();
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float lse = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
        float v[32];
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            if (nb > 0)
                tld32(tlO + 32 * c, v);
            else
#pragma unroll
                for (int k = 0; k < 32; ++k) v[k] = 0.f;
            if (i < rows) {
                if constexpr (DEC) {
                    float* dst = a.po + ((int64_t)i7 + i) * D + 32 * c;
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        *reinterpret_cast<float4*>(dst + k) =
                            make_float4(v[k] * inv, v[k + 1] * inv, v[k + 2] * inv, v[k + 3] * inv);
                } else {
                    const int64_t orow = ((int64_t)i6 + i / a.G) * a.Hq + kvh * a.G + i % a.G;
                    bf16* dst = a.o + orow * D + 32 * c;
#pragma unroll
                    for (int k = 0; k < 32; k += 8)
                        *reinterpret_cast<uint4*>(dst + k) =
                            make_uint4(pack_bf16(v[k] * inv, v[k + 1] * inv), pack_bf16(v[k + 2] * inv, v[k + 3] * inv),
                                       pack_bf16(v[k + 4] * inv, v[k + 5] * inv),
                                       pack_bf16(v[k + 6] * inv, v[k + 7] * inv));
                }
            }
        }
        if (i < rows) {
            if constexpr (DEC)
                a.plse[(int64_t)i7 + i] = lse;
            else
                a.lse[((int64_t)i6 + i / a.G) * a.Hq + kvh * a.G + i % a.G] = lse;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;\n" ::"r"(tbase));
    }
}

template <int D, bool DEC>
int tc_prepare() {
    static int attr = (int)cudaFuncSetAttribute(tc_attn_kernel<D, DEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                TcLayout<D>::TOTAL);
    return attr;
}

}  // namespace

// Extend over all requests: grid (tiles of 128/G new tokens, KV heads).
template <int D>
int launch_extend_tc(const void* q, const void* kp, const void* vp, const int32_t* r2t, int64_t ld,
                     const int32_t* pre, const int32_t* ext, int B, int64_t n_rows, int64_t tiles, void* o, float* lse,
                     uint32_t* err, int Hq, int Hkv, int64_t num_slots, float scale_log2, cudaStream_t s) {
    int e = tc_prepare<D, false>();
    if (e) return e;
    TcArgs a{};
    a.q = static_cast<const bf16*>(q);
    a.kp = static_cast<const bf16*>(kp);
    a.vp = static_cast<const bf16*>(vp);
    a.r2t = r2t;
    a.ld = ld;
    a.prefix_lens = pre;
    a.extend_lens = ext;
    a.B = B;
    a.n_rows = n_rows;
    a.o = static_cast<bf16*>(o);
    a.lse = lse;
    a.err = err;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.num_slots = num_slots;
    a.scale_log2 = scale_log2;
    tc_attn_kernel<D, false><<<dim3((unsigned)tiles, (unsigned)Hkv), kTcThreads, TcLayout<D>::TOTAL, s>>>(a);
    return (int)cudaGetLastError();
}

// Wide decode items (at most 128 query rows each) -> partial rows.
template <int D>
int launch_decode_wide_tc(const DecItem* items, int n_items, const void* q, const void* kp, const void* vp,
                          const int32_t* r2t, int64_t ld, const int32_t* seq_lens, const int32_t* members, float* po,
                          float* plse, uint32_t* err, int Hq, int Hkv, int64_t num_slots, float scale_log2,
                          cudaStream_t s) {
    if (n_items <= 0) return 0;
    int e = tc_prepare<D, true>();
    if (e) return e;
    TcArgs a{};
    a.q = static_cast<const bf16*>(q);
    a.kp = static_cast<const bf16*>(kp);
    a.vp = static_cast<const bf16*>(vp);
    a.r2t = r2t;
    a.ld = ld;
    a.seq_lens = seq_lens;
    a.items = items;
    a.members = members;
    a.po = po;
    a.plse = plse;
    a.err = err;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.num_slots = num_slots;
    a.scale_log2 = scale_log2;
    tc_attn_kernel<D, true><<<n_items, kTcThreads, TcLayout<D>::TOTAL, s>>>(a);
    return (int)cudaGetLastError();
}

template int launch_extend_tc<64>(const void*, const void*, const void*, const int32_t*, int64_t, const int32_t*,
                                  const int32_t*, int, int64_t, int64_t, void*, float*, uint32_t*, int, int, int64_t,
                                  float, cudaStream_t);
template int launch_extend_tc<128>(const void*, const void*, const void*, const int32_t*, int64_t, const int32_t*,
                                   const int32_t*, int, int64_t, int64_t, void*, float*, uint32_t*, int, int, int64_t,
                                   float, cudaStream_t);
template int launch_decode_wide_tc<64>(const DecItem*, int, const void*, const void*, const void*, const int32_t*,
                                       int64_t, const int32_t*, const int32_t*, float*, float*, uint32_t*, int, int,
                                       int64_t, float, cudaStream_t);
template int launch_decode_wide_tc<128>(const DecItem*, int, const void*, const void*, const void*, const int32_t*,
                                        int64_t, const int32_t*, const int32_t*, float*, float*, uint32_t*, int, int,
                                        int64_t, float, cudaStream_t);

}  // namespace sgl
