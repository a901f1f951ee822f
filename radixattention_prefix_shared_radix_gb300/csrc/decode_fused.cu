// Decode attention (bf16): one persistent launch for all partials, then the
// log-sum-exp merge launch.
//
// "SGLang 深度拆解" (chenxutan.com/d/5669.html) §3.2 PagedDecode: one query
// token per request against its whole KV history, gathered through
// req_to_token; memory-bound.  The prefix groups of the batch ("SGLang：从前端
// DSL 到 SRT 服务运行时", section "用基数树实现前缀复用": a shared prefix is
// stored once and referenced by every request that shares it) decide what is
// read once: a segment shared by many requests is read once for all of them.
//
// One CTA per SM (the planner's n_ctas), 480 threads:
//   warps 0-6   the tcgen05 tile roles (tc_tile.cuh) over this CTA's wide
//               items: a chunk of a shared segment against up to 128 query
//               rows (member request x query head of one KV head);
//   warps 7-10  streaming producers: each issues the cp.async gathers of one
//               consumer's K/V rows into its shared-memory ring;
//   warps 11-14 streaming consumers: each runs its own list of narrow items
//               (at most 8 query rows: one request's G heads, or a few
//               members of a small group) on the tensor cores.
// The tiles are bound by latency and the tensor pipe, the streams by HBM; the
// two run side by side on every SM.  Producers and consumers are separate
// warps so the copies keep flowing while the consumers compute, and there is
// one producer per consumer: measured on GB300, a warp issuing random
// 256-byte-row cp.async gathers gets one instruction through every ~80-100
// cycles once the SM's load pipe is busy, so the SM's issue rate (and HBM
// bandwidth) grows with the number of issuing warps.
//
// Streaming ring per consumer: 4 stages of 16 positions (K and V rows, 8 KB),
// a FULL mbarrier per stage (each producer lane arrives when its copies have
// landed: cp.async.mbarrier.arrive.noinc) and an EMPTY mbarrier (the consumer
// arrives when it has read the stage).  The producer looks slots up six steps
// ahead with 4-byte cp.async into a small slot ring, so no register ever
// waits on a load in flight; its own cp.async groups order slot lookups
// before their use.
//
// Consumer, per 16-position step (mma.sync m16n8k16, bf16 in, fp32 acc;
// query rows in the MMA's N dimension):
//   S^T [16 pos x 8 rows] = K [16 x d] . Q^T [d x 8 rows]
//   O^T [d x 8 rows]     += V^T [d x 16 pos] . P^T [16 pos x 8 rows]
// K and V rows are XOR-swizzled [16 x d] tiles (ldmatrix for K,
// ldmatrix.trans for V^T, conflict-free); P^T moves from the accumulator
// layout to the B-operand layout with movmatrix.  The next item's query rows
// are fetched while the current item runs.
//
// Every item writes normalised partial rows (O fp32, LSE natural log); the
// merge launch (merge.cuh) combines each (request, KV head)'s partials once
// all are written, when HBM is idle and each merge is a few short round
// trips.

#include "merge.cuh"
#include "tc_tile.cuh"

namespace sgl {
namespace {

using namespace sgldev;
using namespace tc;

constexpr int kConsumers = kDecNarrowWarps;              // streaming consumer warps per CTA
constexpr int kProducers = kConsumers;                   // one per consumer
constexpr int kNS = 4;                                   // ring stages per consumer
constexpr int kNP = 16;                                  // KV positions per step
constexpr int kQD = 6;                                   // slot lookups ahead (steps per consumer)
constexpr int kSQ = 8;                                   // slot ring entries per consumer
constexpr int kFirstProducer = kTileThreads / 32;
constexpr int kFirstConsumer = kFirstProducer + kProducers;
constexpr int kFusedThreads = 32 * (kFirstConsumer + kConsumers);
static_assert(kSQ >= kQD && (kSQ & (kSQ - 1)) == 0, "slot ring");

template <int D>
struct FusedLayout {
    using TL = TcLayout<D, true>;
    static constexpr int TILEB = kNP * D * 2;            // one K (or V) tile of a step
    static constexpr int STAGE = 2 * TILEB;
    static constexpr int RING = kNS * STAGE;             // per consumer
    static constexpr int SLOTW = kSQ * kNP * 4 + kSQ * 4;   // slots + KV heads per consumer
    static constexpr int OFF_RING = (TL::END + 127) / 128 * 128;
    static constexpr int OFF_SLOT = OFF_RING + kConsumers * RING;
    static constexpr int OFF_SBAR = OFF_SLOT + kConsumers * SLOTW;   // FULL[kNS], EMPTY[kNS] per consumer
    static constexpr int END = OFF_SBAR + kConsumers * 2 * kNS * 8;
    static constexpr int TOTAL = END + 1024;             // + alignment slack
    static_assert(TOTAL <= 232448, "shared memory per CTA");
};

struct FusedArgs {
    TcArgs t;
    const int32_t* wptr;   // [n_ctas + 1] wide items of each CTA
    const int32_t* nptr;   // [n_ctas * kConsumers + 1] narrow items of each consumer
};

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// Fields of a warp's items, lane k holding item it0 + k (at most 32 items).
struct ItemFields {
    int row = 0, b = 0, e = 0, h = 0, mb = 0, nm = 0, pb = 0;
    __device__ __forceinline__ void load(const DecItem* items, int it0, int n_it, int lane) {
        if (lane < n_it) {
            const int4* ip = reinterpret_cast<const int4*>(items + it0 + lane);
            const int4 x = __ldg(ip), y = __ldg(ip + 1);
            row = x.x;
            b = x.y;
            e = x.z;
            h = x.w;
            mb = y.x;
            nm = y.y;
            pb = y.z;
        }
    }
};

__device__ __forceinline__ int fld(int v, int k) { return __shfl_sync(0xffffffffu, v, k); }

__device__ __forceinline__ int total_steps(const ItemFields& it, int n_it, int lane) {
    int s = lane < n_it ? (it.e - it.b + kNP - 1) / kNP : 0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
}

// ---------------------------------------------------------------------------
// Producer: NCP consumers' rings, steps interleaved
// ---------------------------------------------------------------------------
struct SlotCursor {        // the next step of one consumer whose slots are looked up
    int si, sp, n;         // item, position, steps looked up so far
};

template <int D, int NCP>
__device__ __noinline__ void stream_producer(const FusedArgs& f, const int (&it0)[NCP], const int (&n_it)[NCP],
                                             const uint32_t (&ring)[NCP], const uint32_t (&sring)[NCP],
                                             const uint32_t (&full)[NCP], const uint32_t (&empty)[NCP], int lane) {
    using Lay = FusedLayout<D>;
    constexpr int CPR = D / 8;                 // 16-byte chunks per row
    constexpr int RPI = 32 / CPR;              // rows per warp instruction
    constexpr int32_t kPastEnd = INT32_MIN;
    // argument fields in registers: every cp.async below clobbers memory
    const bf16* const kp = f.t.kp;
    const bf16* const vp = f.t.vp;
    const int32_t* const r2t = f.t.r2t;
    const int64_t ld = f.t.ld;
    uint32_t* const err = f.t.err;
    const int Hkv = f.t.Hkv;
    const int64_t num_slots = f.t.num_slots;

    ItemFields it[NCP];
    int steps[NCP];
    SlotCursor cur[NCP];
#pragma unroll
    for (int c = 0; c < NCP; ++c) {
        it[c].load(f.t.items, it0[c], n_it[c], lane);
        steps[c] = total_steps(it[c], n_it[c], lane);
        cur[c] = {0, fld(it[c].b, 0), 0};
        while (cur[c].si < n_it[c] && cur[c].sp >= fld(it[c].e, cur[c].si)) {
            ++cur[c].si;
            if (cur[c].si < n_it[c]) cur[c].sp = fld(it[c].b, cur[c].si);
        }
    }
    // slots of consumer c's next step into its slot ring (kPastEnd beyond the
    // item), its KV head into the head ring (-1: no step)
    auto look_up = [&](int c) {
        SlotCursor& q = cur[c];
        const int ent = q.n & (kSQ - 1);
        const uint32_t hring = sring[c] + kSQ * kNP * 4;
        int kvh = -1;
        if (q.si < n_it[c]) {
            const int row = fld(it[c].row, q.si), e = fld(it[c].e, q.si);
            kvh = fld(it[c].h, q.si);
            const int p = q.sp + lane;
            const uint32_t dst = sring[c] + (ent * kNP + lane) * 4;
            if (lane < kNP) {
                if (p < e)
                    cp_async4(dst, r2t + (int64_t)row * ld + p);
                else
                    st_shared_s32(dst, kPastEnd);
            }
            q.sp += kNP;
            while (q.si < n_it[c] && q.sp >= fld(it[c].e, q.si)) {
                ++q.si;
                if (q.si < n_it[c]) q.sp = fld(it[c].b, q.si);
            }
        }
        if (lane == 0) st_shared_s32(hring + ent * 4, kvh);
        ++q.n;
    };
    for (int k = 0; k < kQD; ++k)
#pragma unroll
        for (int c = 0; c < NCP; ++c) look_up(c);
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();

    // Round r issues step r of each consumer (one cp.async group each, empty
    // once a consumer has no steps left, so the group count stays regular:
    // the lookup of (c, r) is in the group committed NCP*kQD groups earlier).
    bool timed_out = false;
    int rounds = 0;
#pragma unroll
    for (int c = 0; c < NCP; ++c) rounds = steps[c] > rounds ? steps[c] : rounds;
    for (int r = 0; r < rounds; ++r) {
#pragma unroll
        for (int c = 0; c < NCP; ++c) {
            cp_async_wait<NCP * kQD - 1>();
            __syncwarp();
            if (r < steps[c]) {
                const int st = r % kNS;
                if (!timed_out && !mbar_wait_sleep(empty[c] + 8 * st, ((r / kNS) & 1) ^ 1)) {
                    atomicOr(err, 4u);
                    timed_out = true;
                }
                const int ent = r & (kSQ - 1);
                const int kvh = ld_shared_s32(sring[c] + kSQ * kNP * 4 + ent * 4);
                int32_t sl = lane < kNP ? ld_shared_s32(sring[c] + (ent * kNP + lane) * 4) : kPastEnd;
                if (sl == kPastEnd) {
                    sl = -1;
                } else if (sl < 0 || sl >= num_slots) {
                    atomicOr(err, 1u);
                    sl = -1;
                }
                const uint32_t kd = ring[c] + st * Lay::STAGE, vd = kd + Lay::TILEB;
                const int ch = lane % CPR;
#pragma unroll
                for (int k = 0; k < kNP / RPI; ++k) {
                    const int rl = k * RPI + lane / CPR;
                    const int32_t sr = __shfl_sync(0xffffffffu, sl, rl);
                    const int64_t off = sr >= 0 ? ((int64_t)sr * Hkv + (kvh < 0 ? 0 : kvh)) * D + ch * 8 : 0;
                    cp_async16(kd + swz<D>(rl, ch), kp + off, sr >= 0);
                    cp_async16(vd + swz<D>(rl, ch), vp + off, sr >= 0);
                }
                cp_async_arrive_noinc(full[c] + 8 * st);
            }
            __syncwarp();   // every lane has read entry r before it is refilled
            look_up(c);     // step r + kQD
            cp_async_commit();
        }
    }
    cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// Consumer
// ---------------------------------------------------------------------------
template <int D>
__device__ __noinline__ void stream_consumer(const FusedArgs& f, int it0, int n_it, uint32_t ring, uint32_t full,
                                             uint32_t empty, int lane) {
    using Lay = FusedLayout<D>;
    constexpr int MT = D / 16;                 // m-tiles of O^T
    const int g = lane >> 2, t = lane & 3;
    const bf16* const qp = f.t.q;
    const int32_t* const members = f.t.members;
    const int32_t* const seq_lens = f.t.seq_lens;
    float* const po = f.t.po;
    float* const plse = f.t.plse;
    uint32_t* const err = f.t.err;
    const int Hq = f.t.Hq, G = f.t.G;
    const float sc = f.t.scale_log2;

    // it.e is the planned end (steps are counted on it), f_ec the end clamped
    // to the row's seq_len (masks); the clamp does not hold up anything else
    ItemFields it;
    it.load(f.t.items, it0, n_it, lane);
    const int total = total_steps(it, n_it, lane);
    int f_ec = it.e;
    if (lane < n_it) {
        const int len = __ldg(seq_lens + it.row);
        if (it.e > len) {
            atomicOr(err, 2u);
            f_ec = len > it.b ? len : it.b;
        }
    }

    // query rows: the next item's member index is loaded one step before its
    // query words, so neither load stalls the warp
    uint32_t qcur[D / 8], qnext[D / 8];
    int mnext = 0, m_item = -1, q_item = -1;
    auto q_member = [&](int k) {   // phase 1: member request of row g of item k
        if (k < n_it) {
            const int rows = fld(it.nm, k) * G, mb = fld(it.mb, k);
            mnext = g < rows ? __ldg(members + mb + g / G) : -1;
            m_item = k;
        }
    };
    auto q_words = [&]() {         // phase 2: its query words into qnext
        if (m_item < 0) return;
        const int kvh = fld(it.h, m_item);
        const bool ok = mnext >= 0;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            qp + ((int64_t)(ok ? mnext : 0) * Hq + kvh * G + g % G) * D);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qnext[2 * ks] = ok ? __ldg(qrow + 8 * ks + t) : 0u;
            qnext[2 * ks + 1] = ok ? __ldg(qrow + 8 * ks + 4 + t) : 0u;
        }
        q_item = m_item;
        m_item = -1;
    };
    q_member(0);

    float o[MT][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    auto start_item = [&](int k) {
#pragma unroll
        for (int i = 0; i < MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
        if (q_item != k) q_words();   // item k's member index is in flight (short previous item)
#pragma unroll
        for (int w = 0; w < D / 8; ++w) qcur[w] = qnext[w];
        q_member(k + 1);
    };
    auto finish_item = [&](int k) {
        const int rows = fld(it.nm, k) * G, pb = fld(it.pb, k);
        float s0 = l0, s1 = l1;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, off);
            s1 += __shfl_xor_sync(0xffffffffu, s1, off);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = 2 * t + h;
            if (r < rows) {
                const float ll = h ? s1 : s0, mm = h ? m1 : m0;
                const float inv = ll > 0.f ? 1.f / ll : 0.f;
                float* dst = po + ((int64_t)pb + r) * D + g;
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    dst[16 * i] = o[i][h] * inv;
                    dst[16 * i + 8] = o[i][2 + h] * inv;
                }
                if (g == 0) plse[(int64_t)pb + r] = ll > 0.f ? (mm + log2f(ll)) * kLn2 : -INFINITY;
            }
        }
    };

    int ci = 0;
    start_item(0);
    while (ci < n_it && fld(it.e, ci) <= fld(it.b, ci)) {   // leading empty items
        finish_item(ci);
        ++ci;
        if (ci < n_it) start_item(ci);
    }
    int cp0 = ci < n_it ? fld(it.b, ci) : 0;
    int ce = ci < n_it ? fld(it.e, ci) : 0, cm = ci < n_it ? fld(f_ec, ci) : 0;
    bool timed_out = false;
    for (int c = 0; c < total; ++c) {
        const int st = c % kNS;
        if (!timed_out && !mbar_wait_sleep(full + 8 * st, (c / kNS) & 1)) {
            atomicOr(err, 4u);
            timed_out = true;
        }
        // ---- one step of item ci at positions cp0 .. cp0+15
        const uint32_t kb = ring + st * Lay::STAGE, vb = kb + Lay::TILEB;
        // two accumulators halve the dependent MMA chain
        float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t ka[4];
            const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
            ldsm_x4(kb + swz<D>(row, 2 * ks + (lane >> 4)), ka[0], ka[1], ka[2], ka[3]);
            mma16816((ks & 1) ? s2 : s, ka, qcur[2 * ks], qcur[2 * ks + 1]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) s[k] += s2[k];
        const bool ok0 = cp0 + g < cm, ok1 = cp0 + g + 8 < cm;
        s[0] = ok0 ? s[0] * sc : -INFINITY;
        s[1] = ok0 ? s[1] * sc : -INFINITY;
        s[2] = ok1 ? s[2] * sc : -INFINITY;
        s[3] = ok1 ? s[3] * sc : -INFINITY;
        float x0 = fmaxf(s[0], s[2]), x1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
        }
        // Lazy rescale: the running max used for P moves only when a row's
        // block max exceeds it by more than 8 (a factor 2^8, harmless in
        // fp32), so after the first steps O is rarely rescaled.
        const bool up0 = x0 > m0 + 8.f, up1 = x1 > m1 + 8.f;
        if (__any_sync(0xffffffffu, up0 || up1)) {
            const float n0 = up0 ? x0 : m0, n1 = up1 ? x1 : m1;
            const float al0 = m0 == -INFINITY ? 0.f : exp2f(m0 - n0), al1 = m1 == -INFINITY ? 0.f : exp2f(m1 - n1);
            m0 = n0;
            m1 = n1;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                o[i][0] *= al0;
                o[i][1] *= al1;
                o[i][2] *= al0;
                o[i][3] *= al1;
            }
        }
        const float u0 = m0 == -INFINITY ? 0.f : m0, u1 = m1 == -INFINITY ? 0.f : m1;
        const float p00 = exp2f(s[0] - u0), p01 = exp2f(s[1] - u1);
        const float p10 = exp2f(s[2] - u0), p11 = exp2f(s[3] - u1);
        l0 += p00 + p10;
        l1 += p01 + p11;
        const uint32_t pb0 = movtrans(pack_bf16(p00, p01));
        const uint32_t pb1 = movtrans(pack_bf16(p10, p11));
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            uint32_t va[4];
            const int row = (lane & 7) + (lane >> 4) * 8;
            ldsm_x4_t(vb + swz<D>(row, 2 * i + ((lane >> 3) & 1)), va[0], va[1], va[2], va[3]);
            mma16816(o[i], va, pb0, pb1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + 8 * st);   // the stage may be refilled
        if (m_item >= 0) q_words();   // one step after the member index was requested
        cp0 += kNP;
        if (cp0 >= ce) {
            finish_item(ci);
            ++ci;
            while (ci < n_it) {
                start_item(ci);
                if (fld(it.e, ci) > fld(it.b, ci)) break;
                finish_item(ci);   // empty item: LSE -inf partial
                ++ci;
            }
            if (ci < n_it) {
                cp0 = fld(it.b, ci);
                ce = fld(it.e, ci);
                cm = fld(f_ec, ci);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Tile roles: the CTA's wide items
// ---------------------------------------------------------------------------
__device__ __forceinline__ void dec_tile_info(const TcArgs& a, int w, int* info) {
    const DecItem it = a.items[w];
    int e = it.kv_end;
    const int len = __ldg(a.seq_lens + it.rep_row);
    if (e > len) {
        atomicOr(a.err, 2u);
        e = len;
    }
    info[0] = it.rep_row;
    info[1] = it.kv_begin;
    info[2] = e > it.kv_begin ? e : it.kv_begin;
    info[3] = it.kvh;
    info[4] = it.n_mem * a.G;
    info[5] = it.mem_begin;
    info[6] = it.partial_base;
}

template <int D>
__global__ void __maxnreg__(128) decode_fused_kernel(const __grid_constant__ FusedArgs f) {
    using Lay = FusedLayout<D>;
    using TL = TcLayout<D, true>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int w0 = __ldg(f.wptr + blockIdx.x), w1 = __ldg(f.wptr + blockIdx.x + 1);
    const bool tiles = w1 > w0;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + TL::OFF_TMEM);
    int* info = reinterpret_cast<int*>(sm + TL::OFF_INFO);
    const uint32_t sbar = smem_u32(sm + Lay::OFF_SBAR);
    auto full_of = [&](int c) { return sbar + (uint32_t)(c * 2 * kNS) * 8; };
    auto empty_of = [&](int c) { return sbar + (uint32_t)(c * 2 * kNS + kNS) * 8; };
    if (tid == 0) {
        if (tiles) tc_init_barriers<D, true>(smem_u32(sm + TL::OFF_BAR));
        for (int c = 0; c < kConsumers; ++c)
            for (int s = 0; s < kNS; ++s) {
                mbar_init(full_of(c) + 8 * s, 32);    // the producer's 32 lanes
                mbar_init(empty_of(c) + 8 * s, 1);    // the consumer
            }
        mbar_fence_init();
    }
    if (tiles && warp == 4) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(tslot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp < kFirstProducer) {
        if (tiles) {
            const uint32_t tbase = *tslot;
            TcState st{0u, 0u, false};
            for (int w = w0; w < w1; ++w) {
                if (tid == 0) dec_tile_info(f.t, w, info);
                named_bar(kTileBar, kTileThreads);
                const TileInfo ti{info[0], info[1], info[2], info[3], info[4], info[5], info[6]};
                tc_tile_run<D, true>(f.t, ti, sm, tbase, st, tid);
                named_bar(kTileBar, kTileThreads);
            }
        }
    } else if (warp < kFirstConsumer) {
        constexpr int NCP = kConsumers / kProducers;
        const int p = warp - kFirstProducer;
        int it0[NCP], n_it[NCP];
        uint32_t ring[NCP], sring[NCP], full[NCP], empty[NCP];
        bool any = false;
#pragma unroll
        for (int k = 0; k < NCP; ++k) {
            const int c = NCP * p + k, gw = blockIdx.x * kConsumers + c;
            it0[k] = __ldg(f.nptr + gw);
            n_it[k] = __ldg(f.nptr + gw + 1) - it0[k];
            ring[k] = smem_u32(sm + Lay::OFF_RING + c * Lay::RING);
            sring[k] = smem_u32(sm + Lay::OFF_SLOT + c * Lay::SLOTW);
            full[k] = full_of(c);
            empty[k] = empty_of(c);
            any |= n_it[k] > 0;
        }
        if (any) stream_producer<D, NCP>(f, it0, n_it, ring, sring, full, empty, lane);
    } else {
        const int c = warp - kFirstConsumer, gw = blockIdx.x * kConsumers + c;
        const int it0 = __ldg(f.nptr + gw), n_it = __ldg(f.nptr + gw + 1) - it0;
        if (n_it > 0)
            stream_consumer<D>(f, it0, n_it, smem_u32(sm + Lay::OFF_RING + c * Lay::RING), full_of(c), empty_of(c),
                               lane);
    }
    tc_fence_before();
    __syncthreads();
    if (tiles && warp == 4) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(*tslot));
    }
}

}  // namespace

template <int D>
int launch_decode_fused(const sgl_plan* plan, const void* q, const void* kp, const void* vp, const int32_t* r2t,
                        int64_t ld, const int32_t* seq_lens, void* o, float* lse, unsigned char* ws, float scale_log2,
                        cudaStream_t s) {
    using Lay = FusedLayout<D>;
    static const int attr = (int)cudaFuncSetAttribute(decode_fused_kernel<D>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::TOTAL);
    if (attr) return attr;
    const sgl_attn_params& p = plan->params;
    FusedArgs f{};
    TcArgs& a = f.t;
    a.q = static_cast<const bf16*>(q);
    a.kp = static_cast<const bf16*>(kp);
    a.vp = static_cast<const bf16*>(vp);
    a.r2t = r2t;
    a.ld = ld;
    a.seq_lens = seq_lens;
    a.items = reinterpret_cast<const DecItem*>(ws + plan->off_items);
    a.members = reinterpret_cast<const int32_t*>(ws + plan->off_members);
    a.po = reinterpret_cast<float*>(ws + plan->off_po);
    a.plse = reinterpret_cast<float*>(ws + plan->off_plse);
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.Hq = p.num_qo_heads;
    a.Hkv = p.num_kv_heads;
    a.G = plan->G;
    a.num_slots = p.num_slots;
    a.scale_log2 = scale_log2;
    f.wptr = reinterpret_cast<const int32_t*>(ws + plan->off_wptr);
    f.nptr = reinterpret_cast<const int32_t*>(ws + plan->off_nptr);
    decode_fused_kernel<D><<<plan->n_ctas, kFusedThreads, Lay::TOTAL, s>>>(f);
    int e = (int)cudaGetLastError();
    if (e) return e;
    MergeArgs m{a.po, a.plse, reinterpret_cast<const int32_t*>(ws + plan->off_mptr),
                reinterpret_cast<const int32_t*>(ws + plan->off_ment), o, lse, a.Hq, a.Hkv, a.G};
    const int n_pairs = p.batch * a.Hkv;
    decode_merge_kernel<bf16, D><<<(n_pairs + 3) / 4, 128, 0, s>>>(m, n_pairs);
    return (int)cudaGetLastError();
}

template int launch_decode_fused<64>(const sgl_plan*, const void*, const void*, const void*, const int32_t*, int64_t,
                                     const int32_t*, void*, float*, unsigned char*, float, cudaStream_t);
template int launch_decode_fused<128>(const sgl_plan*, const void*, const void*, const void*, const int32_t*, int64_t,
                                      const int32_t*, void*, float*, unsigned char*, float, cudaStream_t);

}  // namespace sgl
