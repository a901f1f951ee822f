// Decode attention (bf16) as one persistent launch per call.
//
// "SGLang 深度拆解" (chenxutan.com/d/5669.html) §3.2 PagedDecode: one query
// token per request against its whole KV history, gathered through
// req_to_token; memory-bound.  The prefix groups of the batch ("SGLang：从前端
// DSL 到 SRT 服务运行时", section "用基数树实现前缀复用": a shared prefix is
// stored once and referenced by every request that shares it) decide what is
// read once: a segment shared by many requests is read once for all of them.
//
// One CTA per SM (the planner's n_ctas), 384 threads:
//   warps 0-6   the tcgen05 tile roles (tc_tile.cuh) over this CTA's wide
//               items: a chunk of a shared segment against up to 128 query
//               rows (member request x query head of one KV head);
//   warps 7-11  streaming warps, each over its own list of narrow items (at
//               most 8 query rows: one request's G heads, or a few members of
//               a small group), with a private cp.async ring in shared
//               memory: 4 stages of 8 KB beside a tile's 64 KB, 5 stages in a
//               CTA without tiles.
// The two kinds run side by side on every SM: the tiles are bound by latency
// and the tensor pipe, the streams by HBM.  Measured on GB300 for random
// 256-byte rows: one warp issues cp.async gathers at ~11 GB/s at most, and a
// warp needs ~3 steps (24 KB) in flight to cover the loaded HBM latency, so
// five warps with 4-stage rings (~160 KB of shared memory) per SM is what
// the shared memory left beside a tile can hold.
//
// Streaming warp, per 16-position step of an item (mma.sync m16n8k16, bf16 in,
// fp32 accumulate; query rows in the MMA's N dimension):
//   S^T [16 pos x 8 rows] = K [16 x d] . Q^T [d x 8 rows]
//   O^T [d x 8 rows]     += V^T [d x 16 pos] . P^T [16 pos x 8 rows]
// K and V rows land by 16-byte cp.async in XOR-swizzled [16 x d] tiles
// (ldmatrix for K, ldmatrix.trans for V^T, conflict-free); P^T moves from the
// accumulator layout to the B-operand layout with movmatrix.  Slots are looked
// up four steps ahead of the copies (4-byte cp.async into a small slot ring,
// so no register ever waits on a load in flight) and the copies a ring's
// depth minus one ahead of the MMAs, across item boundaries, so a warp keeps
// its copies in flight from its first step to its last.  Nothing on the way
// to the first copy waits for more than the item table and one slot lookup;
// the next item's query rows are fetched while the current item runs.
//
// Every item writes normalised partial rows (O fp32, LSE natural log).  The
// log-sum-exp merge is fused: each (request, KV head) has a counter in the
// workspace; a producer publishes its rows (threadfence), increments the
// counters of its member requests, and the producer that completes a count
// merges that (request, KV head) (merge.cuh) and resets the counter to zero
// for the next call.  Streaming warps defer their merges to the end of their
// list so the stream is not interrupted.

#include "merge.cuh"
#include "tc_tile.cuh"

namespace sgl {
namespace {

using namespace sgldev;
using namespace tc;

constexpr int kNarrowWarps = kDecNarrowWarps;
constexpr int kNST = 4;                                  // ring stages per streaming warp, CTA with tiles
constexpr int kNSF = 5;                                  // ring stages per streaming warp, CTA without
constexpr int kQD = 4;                                   // slot lookups in flight per streaming warp
constexpr int kNP = 16;                                  // KV positions per step
constexpr int kFusedThreads = kTileThreads + 32 * kNarrowWarps;

template <int D>
struct FusedLayout {
    using TL = TcLayout<D, true>;
    static constexpr int TILEB = kNP * D * 2;            // one K (or V) tile of a step
    static constexpr int STAGE = 2 * TILEB;
    static constexpr int RING_T = kNST * STAGE;          // per streaming warp, beside the tile roles
    static constexpr int RING_F = kNSF * STAGE;          // per streaming warp, CTA without tiles
    static constexpr int OFF_RING_T = (TL::END + 127) / 128 * 128;
    static constexpr int END_T = OFF_RING_T + kNarrowWarps * RING_T;
    static constexpr int END_F = kNarrowWarps * RING_F;
    static constexpr int SQ = kQD;                       // slot ring entries per streaming warp
    static constexpr int SLOTW = SQ * kNP * 4 + SQ * 4;  // slots + KV heads of the entries
    static constexpr int OFF_SLOT = END_T > END_F ? END_T : END_F;
    static constexpr int TOTAL = OFF_SLOT + kNarrowWarps * SLOTW + 1024;   // + alignment slack
    static_assert(TOTAL <= 232448, "shared memory per CTA");
    static_assert((SQ & (SQ - 1)) == 0 && kQD >= kNST - 1 && kQD >= kNSF - 1, "slot ring");
};

struct FusedArgs {
    TcArgs t;
    MergeArgs m;
    const int32_t* wptr;   // [n_ctas + 1] wide items of each CTA
    const int32_t* nptr;   // [n_ctas * kNarrowWarps + 1] narrow items of each streaming warp
    uint32_t* cnt;         // [B * Hkv] merge counters (zero between calls)
    int n_pairs;           // B * Hkv
};

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// Count one finished partial of pair idx = (request, KV head); true for the
// producer that completes the count (it then owns the merge; the counter is
// reset for the next call).  The pair's entry range is loaded alongside the
// atomic and returned for the merge.
__device__ __forceinline__ bool arrive_pair(const FusedArgs& f, int idx, int& e0, int& E) {
    e0 = __ldg(f.m.mptr + idx);
    E = __ldg(f.m.mptr + idx + 1) - e0;
    const uint32_t old = atomicAdd(f.cnt + idx, 1u);
    if (old + 1 == (uint32_t)E) {
        f.cnt[idx] = 0u;
        return true;
    }
    return false;
}

// ---------------------------------------------------------------------------
// Streaming warp
// ---------------------------------------------------------------------------
template <int D, int NS>
__device__ __noinline__ void stream_items(const FusedArgs& f, int it0, int n_it, uint32_t ring, uint32_t sring,
                                          int lane) {
    using Lay = FusedLayout<D>;
    constexpr int CPR = D / 8;                 // 16-byte chunks per row
    constexpr int RPI = 32 / CPR;              // rows per warp instruction
    constexpr int MT = D / 16;                 // m-tiles of O^T
    constexpr int SQ = Lay::SQ;                // slot ring entries (steps)
    const int g = lane >> 2, t = lane & 3;
    // argument fields in registers: every cp.async below clobbers memory, so
    // fields read through the argument reference would be reloaded each time
    const bf16* const kp = f.t.kp;
    const bf16* const vp = f.t.vp;
    const bf16* const qp = f.t.q;
    const int32_t* const r2t = f.t.r2t;
    const int64_t ld = f.t.ld;
    const int32_t* const members = f.t.members;
    const int32_t* const seq_lens = f.t.seq_lens;
    float* const po = f.t.po;
    float* const plse = f.t.plse;
    uint32_t* const err = f.t.err;
    const int Hq = f.t.Hq, Hkv = f.t.Hkv, G = f.t.G;
    const int64_t num_slots = f.t.num_slots;
    const float sc = f.t.scale_log2;
    const DecItem* const items = f.t.items;

    // lane k holds the fields of item it0 + k; f_e is the planned end (steps
    // are counted on it), f_ec the end clamped to the row's seq_len (masks)
    int f_row = 0, f_b = 0, f_e = 0, f_h = 0, f_mb = 0, f_nm = 0, f_pb = 0;
    if (lane < n_it) {
        const int4* ip = reinterpret_cast<const int4*>(items + it0 + lane);
        const int4 x = __ldg(ip), y = __ldg(ip + 1);
        f_row = x.x;
        f_b = x.y;
        f_e = x.z;
        f_h = x.w;
        f_mb = y.x;
        f_nm = y.y;
        f_pb = y.z;
    }
    auto fld = [&](int v, int k) { return __shfl_sync(0xffffffffu, v, k); };
    int total = lane < n_it ? (f_e - f_b + kNP - 1) / kNP : 0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);

    // ---- slot cursor.  Step n's slots go to entry n % SQ of this warp's slot
    // ring by 4-byte cp.async (lanes 0..15: positions sp + lane; kPastEnd
    // beyond the item) and its KV head to the head ring (-1: no step).  Nothing
    // waits on these loads in registers; they land with the cp.async group of
    // the step that issued them and are read kQD steps later.
    constexpr int32_t kPastEnd = INT32_MIN;
    const uint32_t hring = sring + SQ * kNP * 4;
    int si = 0, sp = fld(f_b, 0), nlook = 0;
    auto skip_empty = [&]() {
        while (si < n_it && sp >= fld(f_e, si)) {
            ++si;
            if (si < n_it) sp = fld(f_b, si);
        }
    };
    skip_empty();
    auto look_up = [&]() {
        const int ent = nlook & (SQ - 1);
        int kvh = -1;
        if (si < n_it) {
            const int row = fld(f_row, si), e = fld(f_e, si);
            kvh = fld(f_h, si);
            const int p = sp + lane;
            const uint32_t dst = sring + (ent * kNP + lane) * 4;
            if (lane < kNP) {
                if (p < e)
                    cp_async4(dst, r2t + (int64_t)row * ld + p);
                else
                    st_shared_s32(dst, kPastEnd);
            }
            sp += kNP;
            skip_empty();
        }
        if (lane == 0) st_shared_s32(hring + ent * 4, kvh);
        ++nlook;
    };
#pragma unroll 1
    for (int k = 0; k < kQD; ++k) look_up();
    cp_async_commit();

    // seq_len clamp (the slot lookups above do not wait for it)
    int f_ec = f_e;
    if (lane < n_it) {
        const int len = __ldg(seq_lens + f_row);
        if (f_e > len) {
            atomicOr(err, 2u);
            f_ec = len > f_b ? len : f_b;
        }
    }
    cp_async_wait<0>();   // the first kQD steps' slots
    __syncwarp();

    int nprod = 0;
    auto produce = [&]() {
        const int ent = nprod & (SQ - 1);
        const int kvh = ld_shared_s32(hring + ent * 4);
        if (kvh >= 0) {
            int32_t sl = lane < kNP ? ld_shared_s32(sring + (ent * kNP + lane) * 4) : kPastEnd;
            if (sl == kPastEnd) {
                sl = -1;
            } else if (sl < 0 || sl >= num_slots) {
                atomicOr(err, 1u);
                sl = -1;
            }
            const uint32_t kd = ring + (nprod % NS) * Lay::STAGE, vd = kd + Lay::TILEB;
            const int ch = lane % CPR;
#pragma unroll
            for (int k = 0; k < kNP / RPI; ++k) {
                const int rl = k * RPI + lane / CPR;
                const int32_t sr = __shfl_sync(0xffffffffu, sl, rl);
                const int64_t off = sr >= 0 ? ((int64_t)sr * Hkv + kvh) * D + ch * 8 : 0;
                cp_async16(kd + swz<D>(rl, ch), kp + off, sr >= 0);
                cp_async16(vd + swz<D>(rl, ch), vp + off, sr >= 0);
            }
        }
        __syncwarp();      // every lane has read entry `ent` before it is refilled
        look_up();         // step nprod + kQD into the entry just read
        cp_async_commit();
        ++nprod;
    };

    // ---- query rows: the next item's member index is loaded one step before
    // its query words, so neither load stalls the warp
    uint32_t qcur[D / 8], qnext[D / 8];
    int mnext = 0, m_item = -1, q_item = -1;
    auto q_member = [&](int k) {   // phase 1: member request of row g of item k
        if (k < n_it) {
            const int rows = fld(f_nm, k) * G, mb = fld(f_mb, k);
            mnext = g < rows ? __ldg(members + mb + g / G) : -1;
            m_item = k;
        }
    };
    auto q_words = [&]() {         // phase 2: its query words into qnext
        if (m_item < 0) return;
        const int kvh = fld(f_h, m_item);
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
    for (int s = 0; s < NS - 1; ++s) produce();

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
        const int rows = fld(f_nm, k) * G, pb = fld(f_pb, k);
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
    while (ci < n_it && fld(f_e, ci) <= fld(f_b, ci)) {   // leading empty items
        finish_item(ci);
        ++ci;
        if (ci < n_it) start_item(ci);
    }
    int cp0 = ci < n_it ? fld(f_b, ci) : 0;
    int ce = ci < n_it ? fld(f_e, ci) : 0, cm = ci < n_it ? fld(f_ec, ci) : 0;
    for (int c = 0; c < total; ++c) {
        cp_async_wait<NS - 2>();   // step c has landed (and the slots of step c + NS - 1)
        __syncwarp();
        produce();                 // step c + NS - 1
        // ---- one step of item ci at positions cp0 .. cp0+15
        const uint32_t kb = ring + (c % NS) * Lay::STAGE, vb = kb + Lay::TILEB;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t ka[4];
            const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
            ldsm_x4(kb + swz<D>(row, 2 * ks + (lane >> 4)), ka[0], ka[1], ka[2], ka[3]);
            mma16816(s, ka, qcur[2 * ks], qcur[2 * ks + 1]);
        }
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
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
        const float al0 = exp2f(m0 - u0), al1 = exp2f(m1 - u1);
        m0 = n0;
        m1 = n1;
        const float p00 = exp2f(s[0] - u0), p01 = exp2f(s[1] - u1);
        const float p10 = exp2f(s[2] - u0), p11 = exp2f(s[3] - u1);
        l0 = l0 * al0 + p00 + p10;
        l1 = l1 * al1 + p01 + p11;
        const uint32_t pb0 = movtrans(pack_bf16(p00, p01));
        const uint32_t pb1 = movtrans(pack_bf16(p10, p11));
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            o[i][0] *= al0;
            o[i][1] *= al1;
            o[i][2] *= al0;
            o[i][3] *= al1;
            uint32_t va[4];
            const int row = (lane & 7) + (lane >> 4) * 8;
            ldsm_x4_t(vb + swz<D>(row, 2 * i + ((lane >> 3) & 1)), va[0], va[1], va[2], va[3]);
            mma16816(o[i], va, pb0, pb1);
        }
        if (m_item >= 0) q_words();   // one step after the member index was requested
        cp0 += kNP;
        if (cp0 >= ce) {
            finish_item(ci);
            ++ci;
            while (ci < n_it) {
                start_item(ci);
                if (fld(f_e, ci) > fld(f_b, ci)) break;
                finish_item(ci);   // empty item: LSE -inf partial
                ++ci;
            }
            if (ci < n_it) {
                cp0 = fld(f_b, ci);
                ce = fld(f_e, ci);
                cm = fld(f_ec, ci);
            }
        }
    }
    cp_async_wait<0>();
    // Publish this warp's partials once, then count one arrival per (member
    // request, KV head) of every item -- lane p takes the p-th member row
    // (at most 32: the planner caps a warp's member rows) -- and merge the
    // pairs this warp completed.
    __threadfence();
    __syncwarp();
    int idx = -1, p0 = 0;
    for (int k = 0; k < n_it; ++k) {
        const int nm = fld(f_nm, k), mb = fld(f_mb, k), kvh = fld(f_h, k);   // all lanes shuffle
        if (lane >= p0 && lane < p0 + nm) idx = __ldg(members + mb + (lane - p0)) * Hkv + kvh;
        p0 += nm;
    }
    int e0 = 0, E = 0;
    const bool last = idx >= 0 && arrive_pair(f, idx, e0, E);
    unsigned bits = __ballot_sync(0xffffffffu, last);
    if (bits) __threadfence();
    while (bits) {
        const int src = __ffs(bits) - 1;
        bits &= bits - 1;
        merge_warp<bf16, D>(f.m, __shfl_sync(0xffffffffu, idx, src), __shfl_sync(0xffffffffu, e0, src),
                            __shfl_sync(0xffffffffu, E, src), lane);
    }
}

template <int D, int NS>
__device__ __forceinline__ void stream_warp(const FusedArgs& f, int gw, uint32_t ring, uint32_t sring, int lane) {
    const int it0 = __ldg(f.nptr + gw), n_it = __ldg(f.nptr + gw + 1) - it0;
    if (n_it > 0) stream_items<D, NS>(f, it0, n_it, ring, sring, lane);
    // (request, KV head) pairs with no partial at all (seq_len 0)
    const int nwt = gridDim.x * kNarrowWarps;
    for (int idx = gw; idx < f.n_pairs; idx += nwt)
        if (__ldg(f.m.mptr + idx + 1) == __ldg(f.m.mptr + idx)) merge_empty<bf16, D>(f.m, idx, lane);
}

// ---------------------------------------------------------------------------
// Tile roles: decode items of this CTA, then the merges they complete
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
__device__ __forceinline__ void tile_merges(const FusedArgs& f, const TileInfo& ti, uint8_t* sm, int tid) {
    using TL = TcLayout<D, true>;
    int* mcnt = reinterpret_cast<int*>(sm + TL::OFF_MCNT);
    int* mlist = reinterpret_cast<int*>(sm + TL::OFF_MLIST);
    const TcArgs& a = f.t;
    __threadfence();
    named_bar(kSoftmaxBar, 128);
    const int nm = ti.rows / a.G;
    if (tid < nm) {
        const int idx = __ldg(a.members + ti.i6 + tid) * a.Hkv + ti.kvh;
        int e0, E;
        if (arrive_pair(f, idx, e0, E)) mlist[atomicAdd(mcnt, 1)] = idx;
    }
    named_bar(kSoftmaxBar, 128);
    const int n = *mcnt;
    if (n > 0) {
        __threadfence();
        for (int k = tid >> 5; k < n; k += 4) {
            const int idx = mlist[k];
            const int e0 = __ldg(f.m.mptr + idx), E = __ldg(f.m.mptr + idx + 1) - e0;
            merge_warp<bf16, D>(f.m, idx, e0, E, tid & 31);
        }
    }
    named_bar(kSoftmaxBar, 128);
    if (tid == 0) *mcnt = 0;
}

template <int D>
__global__ void __maxnreg__(168) decode_fused_kernel(const __grid_constant__ FusedArgs f) {
    using Lay = FusedLayout<D>;
    using TL = TcLayout<D, true>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int w0 = __ldg(f.wptr + blockIdx.x), w1 = __ldg(f.wptr + blockIdx.x + 1);
    const bool tiles = w1 > w0;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + TL::OFF_TMEM);
    int* info = reinterpret_cast<int*>(sm + TL::OFF_INFO);
    if (tiles) {
        if (tid == 0) {
            tc_init_barriers<D, true>(smem_u32(sm + TL::OFF_BAR));
            mbar_fence_init();
            *reinterpret_cast<int*>(sm + TL::OFF_MCNT) = 0;
        }
        if (warp == 4) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
                smem_u32(tslot)));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp < kTileThreads / 32) {
        if (tiles) {
            const uint32_t tbase = *tslot;
            TcState st{0u, 0u, false};
            for (int w = w0; w < w1; ++w) {
                if (tid == 0) dec_tile_info(f.t, w, info);
                named_bar(kTileBar, kTileThreads);
                const TileInfo ti{info[0], info[1], info[2], info[3], info[4], info[5], info[6]};
                tc_tile_run<D, true>(f.t, ti, sm, tbase, st, tid);
                if (warp < 4) tile_merges<D>(f, ti, sm, tid);
                named_bar(kTileBar, kTileThreads);
            }
        }
    } else {
        const int sw = warp - kTileThreads / 32;
        const int gw = blockIdx.x * kNarrowWarps + sw;
        const uint32_t sring = smem_u32(sm + Lay::OFF_SLOT + sw * Lay::SLOTW);
        if (tiles)
            stream_warp<D, kNST>(f, gw, smem_u32(sm + Lay::OFF_RING_T + sw * Lay::RING_T), sring, lane);
        else
            stream_warp<D, kNSF>(f, gw, smem_u32(sm + sw * Lay::RING_F), sring, lane);
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
    f.m.po = a.po;
    f.m.plse = a.plse;
    f.m.mptr = reinterpret_cast<const int32_t*>(ws + plan->off_mptr);
    f.m.ment = reinterpret_cast<const int32_t*>(ws + plan->off_ment);
    f.m.o = o;
    f.m.lse = lse;
    f.m.Hq = a.Hq;
    f.m.Hkv = a.Hkv;
    f.m.G = a.G;
    f.wptr = reinterpret_cast<const int32_t*>(ws + plan->off_wptr);
    f.nptr = reinterpret_cast<const int32_t*>(ws + plan->off_nptr);
    f.cnt = reinterpret_cast<uint32_t*>(ws + plan->off_cnt);
    f.n_pairs = p.batch * a.Hkv;
    decode_fused_kernel<D><<<plan->n_ctas, kFusedThreads, Lay::TOTAL, s>>>(f);
    return (int)cudaGetLastError();
}

template int launch_decode_fused<64>(const sgl_plan*, const void*, const void*, const void*, const int32_t*, int64_t,
                                     const int32_t*, void*, float*, unsigned char*, float, cudaStream_t);
template int launch_decode_fused<128>(const sgl_plan*, const void*, const void*, const void*, const int32_t*, int64_t,
                                      const int32_t*, void*, float*, unsigned char*, float, cudaStream_t);

}  // namespace sgl
