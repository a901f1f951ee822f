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
//   warps 0-10  (CTAs with wide items) the tcgen05 tile roles of
//               tc_tile.cuh over this CTA's wide items: a chunk of a shared
//               segment against up to 128 query rows (member request x query
//               head of one KV head); warps 5-10 are the tiles' gather team;
//   warps 7-10  streaming producers: each issues the cp.async gathers of one
//               consumer's K/V rows into its shared-memory ring (in CTAs
//               with wide items, once the tiles are done);
//   warps 11-14 streaming consumers: each runs narrow pieces (at most 8
//               query rows: one request's G heads, or a few members of a
//               small group) on the tensor cores: its launch piece, then
//               pieces its producer takes from a run-time counter, so faster
//               SMs stream more and all finish together.
// The tiles are bound by latency and the tensor pipe, the streams by HBM.
// The planner puts the wide items on the first CTAs (as many as balance the
// streaming work); their streaming warps wait at a barrier until the tiles are
// done and then take pieces from the run-time counter, so an SM never runs
// both kinds at once (measured: co-running them cost the streams most of
// their instruction-cache hits).  Producers and consumers are separate
// warps so the copies keep flowing while the consumers compute, and there is
// one producer per consumer: measured on GB300, a warp issuing random
// 256-byte-row cp.async gathers gets one instruction through every ~80-100
// cycles once the SM's load pipe is busy, so the SM's issue rate (and HBM
// bandwidth) grows with the number of issuing warps.
//
// Streaming ring per consumer: 4 stages of 16 positions (K and V rows, 8 KB)
// with a descriptor each (first position, piece, flags), a FULL mbarrier per
// stage (each producer lane arrives when its copies have landed:
// cp.async.mbarrier.arrive.noinc, and lane 0 once more to release the
// descriptor) and an EMPTY mbarrier (the consumer arrives when it has read
// the stage).  The producer looks slots up six steps ahead with 4-byte
// cp.async into a small slot ring, so no register ever waits on a load in
// flight; its own cp.async groups order slot lookups before their use.
//
// Consumer, per 16-position step (mma.sync m16n8k16, bf16 in, fp32 acc;
// query rows in the MMA's N dimension):
//   S^T [16 pos x 8 rows] = K [16 x d] . Q^T [d x 8 rows]
//   O^T [d x 8 rows]     += V^T [d x 16 pos] . P^T [16 pos x 8 rows]
// K and V rows are XOR-swizzled [16 x d] tiles (ldmatrix for K,
// ldmatrix.trans for V^T, conflict-free); P^T moves from the accumulator
// layout to the B-operand layout with movmatrix.  A piece's query rows are
// staged by the producer with the piece's first step (two Q slots, released
// by the consumer through a QEMPTY barrier), so the consumer's loop touches
// nothing but shared memory.
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
constexpr int kNS = 2;                                   // ring stages per consumer (tile CTA: beside the tiles' K/V rings)
constexpr int kNSF = 4;                                  // ring stages per consumer (streaming CTA)
constexpr int kNP = 16;                                  // KV positions per step
constexpr int kQD = 6;                                   // slot lookups ahead (steps per consumer)
constexpr int kSQ = 8;                                   // slot ring entries per consumer
constexpr int kSlotEntry = 128;                         // 16 slots + step and piece fields (see below)
constexpr int kGrabAhead = 4;                            // take the next piece this many steps before the end
constexpr int kFirstProducer = 7;                        // after the tile roles' softmax, MMA and own gather warps
static_assert(DecCfg<128>::kThreads == 32 * (kFirstProducer + kProducers) && DecCfg<64>::kThreads == DecCfg<128>::kThreads,
              "the tile roles' gather team is warps 5 .. 10: two of its own and the four producers");
constexpr int kFirstConsumer = kFirstProducer + kProducers;
constexpr int kFusedThreads = 32 * (kFirstConsumer + kConsumers);
static_assert(kSQ >= kQD && (kSQ & (kSQ - 1)) == 0 && kQD >= kNSF - 1, "slot ring");

template <int D, bool F8 = false>
struct FusedLayout {
    using TL = typename DecCfg<D, F8>::Lay;
    static constexpr int TILEB = kNP * D * (F8 ? 1 : 2);   // one K (or V) tile of a step
    static constexpr int STAGE = 2 * TILEB;
    static constexpr int RING = kNS * STAGE;             // per consumer, beside the tile roles
    static constexpr int RING_F = kNSF * STAGE;          // per consumer, CTA without tiles (from offset 0)
    static constexpr int SLOTW = kSQ * kSlotEntry;       // slot ring per consumer
    // Layout from offset 0: the tile roles' TMEM address and broadcast area
    // (up to TL::KEEP), then the rings of a CTA with tiles, the slot rings,
    // descriptors and Q slots.  These are used only once the CTA's tiles are
    // done, so they overlap the rest of the tile roles' area (TL::KEEP ..
    // TL::END: stages, barriers, staging).  A CTA without tiles puts its
    // deeper rings at offset 0.  The streaming barriers, initialised at
    // launch, come after everything.
    static constexpr int OFF_RING = (TL::KEEP + 127) / 128 * 128;
    static constexpr int END_RINGS = (OFF_RING + kConsumers * RING) > kConsumers * RING_F
                                         ? (OFF_RING + kConsumers * RING) : kConsumers * RING_F;
    static constexpr int OFF_SLOT = END_RINGS;
    static constexpr int QSLOT = 8 * D * 2;              // query rows of one piece (at most 8)
    static constexpr int OFF_DESC = OFF_SLOT + kConsumers * SLOTW;   // kNSF stage descriptors (32 B) per consumer
    static constexpr int OFF_Q = (OFF_DESC + kConsumers * kNSF * 32 + 127) / 128 * 128;   // 2 Q slots per consumer
    static constexpr int END_Q = OFF_Q + kConsumers * 2 * QSLOT;
    // FULL[kNSF], EMPTY[kNSF], QEMPTY[2] per consumer
    static constexpr int OFF_SBAR = ((END_Q > TL::END ? END_Q : TL::END) + 7) / 8 * 8;
    static constexpr int END = OFF_SBAR + kConsumers * (2 * kNSF + 2) * 8;
    static constexpr int TOTAL = END + 1024;             // + alignment slack
    static_assert(OFF_SBAR >= TL::END && OFF_SBAR >= END_Q, "streaming barriers clear of every other area");
    static_assert(TOTAL <= 232448, "shared memory per CTA");
};

struct FusedArgs {
    TcArgs t;
    const int32_t* wptr;   // [n_ctas + 1] wide items of each CTA
    const DecItem* narrow; // narrow pieces, longest first
    int n_narrow;
    int n_init;            // pieces assigned at launch: streaming consumer w starts on piece w
    int n_tile_ctas;       // CTAs 0 .. n_tile_ctas-1 run the wide items first
    uint32_t* sched;       // [2] next piece to hand out, producers finished (restored at the end)
};

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// D[16x8] += A[16x16] * B[16x8], f16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816_f16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16-byte chunk c of row r of an FP8 [16 x D] stage tile (rows of D bytes),
// XOR-swizzled so that the consumer's fragment reads (below) are free of
// bank conflicts for D = 128 (two-way for D = 64).
template <int D>
__device__ __forceinline__ uint32_t fswz(int r, int c) {
    return (uint32_t)(r * D + ((c ^ (D == 128 ? (r & 7) : ((r >> 1) & 3))) << 4));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ void lds128(uint32_t addr, uint32_t* w) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
}
__device__ __forceinline__ void lds64(uint32_t addr, uint32_t* w) {
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];\n" : "=r"(w[0]), "=r"(w[1]) : "r"(addr));
}

// stage descriptor flags
constexpr int kFirst = 1;   // first step of its piece: its query rows are in the stage's Q slot
constexpr int kEnd = 4;     // no more pieces: the consumer stops

// slot-ring entry (one looked-up step): 16 slots, then
constexpr int kEntKvh = 64, kEntP0 = 72, kEntFlags = 76, kEntCm = 80, kEntPb = 84, kEntRows = 88;
constexpr int kEntMem = 96;   // 8 ints: member request of each query row (first step only)
// stage descriptor
constexpr int kDescP0 = 0, kDescFlags = 4, kDescCm = 8, kDescPb = 12, kDescRows = 16, kDescQ = 20;

// ---------------------------------------------------------------------------
// Producer
// ---------------------------------------------------------------------------
// Walks this consumer's pieces (its launch piece, then pieces taken from the
// run-time counter), looks up each step's slots kQD steps ahead (4-byte
// cp.async into the slot ring, with the step's KV head, position and flags,
// and for a first step the piece's partial base, rows, clamped end and the
// member request of each query row), and for each step waits for the ring
// stage to be free, issues the K/V row copies (and, for a first step, the
// piece's query rows into one of two Q slots once the consumer has released
// it), writes the stage descriptor and arrives on the stage's FULL barrier
// (32 lanes when their copies land + lane 0 releasing the descriptor).  The
// next piece is fetched in phases spread over the steps (take a number from
// the counter; load its record; load its members and seq_len), so no register
// waits on a load in flight.
template <int D, int NS, bool F8 = false>
__device__ __noinline__ void stream_producer(const FusedArgs& f, int gw, uint32_t ring, uint32_t sring,
                                             uint32_t desc, uint32_t qbuf, uint32_t full, uint32_t empty,
                                             uint32_t qempty, int lane) {
    using Lay = FusedLayout<D, F8>;
    constexpr int CPR = D / 8;                 // 16-byte chunks per row
    constexpr int RPI = 32 / CPR;              // rows per warp instruction
    constexpr int32_t kPastEnd = INT32_MIN;
    // argument fields in registers: every cp.async below clobbers memory
    const bf16* const kp = f.t.kp;
    const bf16* const vp = f.t.vp;
    const bf16* const qp = f.t.q;
    const int32_t* const r2t = f.t.r2t;
    const int32_t* const members = f.t.members;
    const int32_t* const seq_lens = f.t.seq_lens;
    const int64_t ld = f.t.ld;
    uint32_t* const err = f.t.err;
    const int Hq = f.t.Hq, Hkv = f.t.Hkv, G = f.t.G;
    const int64_t num_slots = f.t.num_slots;
    const DecItem* const pieces = f.narrow;
    const int n_narrow = f.n_narrow;
    uint32_t* const sched = f.sched;
    // streamed K/V rows are read once: evict them from L2 first, which keeps
    // the code, the tables and the partial rows there across calls
    const uint64_t kv_pol = l2_evict_first_policy();

    // next-piece pipeline: 0 take a number, 1 number in flight (lane 0),
    // 2 record in flight, 3 members / seq_len in flight, 4 ready;
    // `none` once the counter ran out
    int nx_id = 0, nx_stage = 0, taken = 0;
    int nx_row = 0, nx_b = 0, nx_e = 0, nx_h = 0, nx_mb = 0, nx_nm = 0, nx_pb = 0, nx_mem = 0, nx_len = 0;
    bool none = false;
    auto load_record = [&]() {
        if (nx_id < n_narrow) {
            const int4* rp = reinterpret_cast<const int4*>(pieces + nx_id);
            const int4 x = __ldg(rp), y = __ldg(rp + 1);
            nx_row = x.x;
            nx_b = x.y;
            nx_e = x.z;
            nx_h = x.w;
            nx_mb = y.x;
            nx_nm = y.y;
            nx_pb = y.z;
        } else {
            none = true;
        }
    };
    // the launch piece: its record is waited for once; its seq_len and
    // members are loaded now and used only when its first step is issued
    const bool launch = gw >= 0 && gw < f.n_init;
    int lp_len = 0, lp_mem = 0, lp_b = 0, lp_e = 0, lp_pb = 0, lp_rows = 0;
    if (launch) {
        nx_id = gw;
        load_record();
        nx_stage = 3;
        lp_len = __ldg(seq_lens + nx_row);
        lp_mem = lane < nx_nm * G ? __ldg(members + nx_mb + lane / G) : 0;
        lp_b = nx_b;
        lp_e = nx_e;
        lp_pb = nx_pb;
        lp_rows = nx_nm * G;
    }
    auto advance = [&]() {
        if (none) return;
        if (nx_stage == 0) {
            if (lane == 0) taken = (int)atomicAdd(sched, 1u);
            nx_stage = 1;
        } else if (nx_stage == 1) {
            nx_id = __shfl_sync(0xffffffffu, taken, 0);
            load_record();
            nx_stage = 2;
        } else if (nx_stage == 2) {
            nx_len = __ldg(seq_lens + nx_row);
            nx_mem = lane < nx_nm * G ? __ldg(members + nx_mb + lane / G) : 0;
            nx_stage = 3;
        } else if (nx_stage == 3) {
            nx_stage = 4;
        }
    };
    if (launch) nx_stage = 4;
    bool launch_entry_pending = launch;

    // slot cursor over the current piece
    bool have = false, done = false;
    bool prologue = true;   // the first kQD lookups: no grab-ahead, which would put the next piece's
                            // dependent loads (counter, record, members) before the first step
    int row = 0, e = 0, h = 0, sp = 0, nlook = 0;
    auto look_up = [&]() {
        const int ent = nlook & (kSQ - 1);
        const uint32_t eb = sring + ent * kSlotEntry;
        int kvh = -1, p0 = 0, flags = 0;
        if (!done && (!have || sp >= e)) {
            while (!none && nx_stage < 4) advance();
            if (none) {
                have = false;
                done = true;
            } else {
                have = true;
                row = nx_row;
                sp = nx_b;
                e = nx_e;
                h = nx_h;
                flags = kFirst;
                if (launch_entry_pending) {
                    launch_entry_pending = false;   // fields come from lp_* when step 0 is issued
                } else {
                    int cm = nx_e;
                    if (nx_e > nx_len) {   // planned beyond seq_len: mask the excess, flag it
                        if (lane == 0) atomicOr(err, 2u);
                        cm = nx_len > nx_b ? nx_len : nx_b;
                    }
                    if (lane == 0) {
                        st_shared_s32(eb + kEntCm, cm);
                        st_shared_s32(eb + kEntPb, nx_pb);
                        st_shared_s32(eb + kEntRows, nx_nm * G);
                    }
                    if (lane < 8) st_shared_s32(eb + kEntMem + 4 * lane, nx_mem);
                }
                nx_stage = 0;
            }
        }
        if (have && !done) {
            kvh = h;
            p0 = sp;
            const int p = sp + lane;
            if (lane < kNP) {
                if (p < e)
                    cp_async4(eb + lane * 4, r2t + (int64_t)row * ld + p);
                else
                    st_shared_s32(eb + lane * 4, kPastEnd);
            }
            sp += kNP;
        }
        if (lane == 0) {
            st_shared_s32(eb + kEntKvh, kvh);
            st_shared_s32(eb + kEntP0, p0);
            st_shared_s32(eb + kEntFlags, flags);
        }
        ++nlook;
        // Take the next number only near the end of the current piece: the
        // counter then runs dry only when the work does, and CTAs that join
        // late (tile CTAs) still find pieces.
        if (!prologue && (nx_stage != 0 || !have || done || (e - sp + kNP - 1) / kNP <= kGrabAhead)) advance();
    };
    // one cp.async group per step's lookup: the first step waits for its
    // own slots only
#pragma unroll 1
    for (int k = 0; k < kQD; ++k) {
        look_up();
        cp_async_commit();
    }
    prologue = false;

    bool timed_out = false;
    int nq = 0;   // pieces started (Q slot uses)
    for (int r = 0;; ++r) {
        // the lookup of step r was committed kQD groups ago
        cp_async_wait<kQD - 1>();
        __syncwarp();
        const int ent = r & (kSQ - 1);
        const uint32_t eb = sring + ent * kSlotEntry;
        const int kvh = ld_shared_s32(eb + kEntKvh);
        const int flags = ld_shared_s32(eb + kEntFlags);
        const int st = r % NS;
        if (!timed_out && !mbar_wait_sleep(empty + 8 * st, ((r / NS) & 1) ^ 1)) {
            atomicOr(err, 4u);
            timed_out = true;
        }
        const uint32_t db = desc + st * 32;
        if (kvh >= 0) {
            int32_t sl = lane < kNP ? ld_shared_s32(eb + lane * 4) : kPastEnd;
            if (sl == kPastEnd) {
                sl = -1;
            } else if (sl < 0 || sl >= num_slots) {
                atomicOr(err, 1u);
                sl = -1;
            }
            const uint32_t kd = ring + st * Lay::STAGE, vd = kd + Lay::TILEB;
            if constexpr (F8) {
                // FP8 rows of D bytes, [16 x D] tiles with swizzled chunks
                constexpr int CPB = D / 16, RPB = 32 / CPB;
                const int chb = lane % CPB;
                const uint8_t* kp8 = reinterpret_cast<const uint8_t*>(kp);
                const uint8_t* vp8 = reinterpret_cast<const uint8_t*>(vp);
#pragma unroll
                for (int k = 0; k < kNP / RPB; ++k) {
                    const int rl = k * RPB + lane / CPB;
                    const int32_t sr = __shfl_sync(0xffffffffu, sl, rl);
                    const int64_t off = sr >= 0 ? ((int64_t)sr * Hkv + kvh) * D + chb * 16 : 0;
                    cp_async16_pol(kd + fswz<D>(rl, chb), kp8 + off, sr >= 0, kv_pol);
                    cp_async16_pol(vd + fswz<D>(rl, chb), vp8 + off, sr >= 0, kv_pol);
                }
            } else {
                const int ch = lane % CPR;
#pragma unroll
                for (int k = 0; k < kNP / RPI; ++k) {
                    const int rl = k * RPI + lane / CPR;
                    const int32_t sr = __shfl_sync(0xffffffffu, sl, rl);
                    const int64_t off = sr >= 0 ? ((int64_t)sr * Hkv + kvh) * D + ch * 8 : 0;
                    cp_async16_pol(kd + swz<D>(rl, ch), kp + off, sr >= 0, kv_pol);
                    cp_async16_pol(vd + swz<D>(rl, ch), vp + off, sr >= 0, kv_pol);
                }
            }
            const int ch = lane % CPR;
            if (flags & kFirst) {
                // the piece's query rows (at most 8) into Q slot nq & 1, swizzled
                const int qs = nq & 1;
                if (!timed_out && !mbar_wait_sleep(qempty + 8 * qs, ((nq >> 1) & 1) ^ 1)) {
                    atomicOr(err, 4u);
                    timed_out = true;
                }
                const bool lp = launch && r == 0;   // the launch piece's first step
                int cm, pb, rows;
                if (lp) {
                    cm = lp_e;
                    if (lp_e > lp_len) {
                        if (lane == 0) atomicOr(err, 2u);
                        cm = lp_len > lp_b ? lp_len : lp_b;
                    }
                    pb = lp_pb;
                    rows = lp_rows;
                } else {
                    cm = ld_shared_s32(eb + kEntCm);
                    pb = ld_shared_s32(eb + kEntPb);
                    rows = ld_shared_s32(eb + kEntRows);
                }
                const uint32_t qd = qbuf + qs * Lay::QSLOT;
#pragma unroll
                for (int k = 0; k < 8 / RPI; ++k) {
                    const int rq = k * RPI + lane / CPR;
                    const bool ok = rq < rows;
                    const int lpm = __shfl_sync(0xffffffffu, lp_mem, rq);
                    const int mem = lp ? lpm : ld_shared_s32(eb + kEntMem + 4 * rq);
                    const bf16* src = ok ? qp + ((int64_t)mem * Hq + kvh * G + rq % G) * D + ch * 8 : qp;
                    cp_async16(qd + swz<D>(rq, ch), src, ok);
                }
                if (lane == 0) {
                    st_shared_s32(db + kDescCm, cm);
                    st_shared_s32(db + kDescPb, pb);
                    st_shared_s32(db + kDescRows, rows);
                    st_shared_s32(db + kDescQ, qs);
                }
                ++nq;
            }
        }
        if (lane == 0) {
            st_shared_s32(db + kDescP0, ld_shared_s32(eb + kEntP0));
            st_shared_s32(db + kDescFlags, kvh >= 0 ? flags : kEnd);
        }
        cp_async_arrive_noinc(full + 8 * st);    // each lane, when its copies have landed
        __syncwarp();
        if (lane == 0) mbar_arrive(full + 8 * st);   // releases the descriptor
        if (kvh < 0) break;
        __syncwarp();   // every lane has read entry r before it is refilled
        look_up();      // step r + kQD
        cp_async_commit();
    }
    cp_async_wait<0>();
    // The last producer to finish restores the counter for the next call
    // (every producer has taken its last number by then).
    if (lane == 0) {
        const uint32_t total = gridDim.x * (uint32_t)kProducers;
        if (atomicAdd(sched + 1, 1u) + 1 == total) {
            sched[0] = (uint32_t)f.n_init;
            sched[1] = 0u;
            __threadfence();
        }
    }
}

// ---------------------------------------------------------------------------
// Consumer: only shared memory in its loop (stages, descriptors, Q slots)
// ---------------------------------------------------------------------------
template <int D, int NS, bool F8 = false>
__device__ __noinline__ void stream_consumer(const FusedArgs& f, uint32_t ring, uint32_t desc, uint32_t qbuf,
                                             uint32_t full, uint32_t empty, uint32_t qempty, int lane) {
    using Lay = FusedLayout<D, F8>;
    constexpr int MT = D / 16;                 // m-tiles of O^T
    const int g = lane >> 2, t = lane & 3;
    float* const po = f.t.po;
    float* const plse = f.t.plse;
    uint32_t* const err = f.t.err;
    // FP8 pools: the K scale goes into the score scale, the V scale into the
    // final normalisation (both are per tensor, so they factor out)
    const float sc = F8 ? f.t.scale_log2 * f.t.k_scale : f.t.scale_log2;
    const float vsc = F8 ? f.t.v_scale : 1.f;

    uint32_t qcur[D / 8];
    float o[MT][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool have = false;
    int cur_pb = 0, cur_rows = 0, cm = 0;
    auto finish_item = [&]() {
        float s0 = l0, s1 = l1;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, off);
            s1 += __shfl_xor_sync(0xffffffffu, s1, off);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = 2 * t + hh;
            if (r < cur_rows) {
                const float ll = hh ? s1 : s0, mm = hh ? m1 : m0;
                const float inv = ll > 0.f ? vsc / ll : 0.f;
                if constexpr (F8) {
                    // m-tile i rows g, g + 8 stand for d = (D/8) g + 2i, + 1
                    float* dst = po + ((int64_t)cur_pb + r) * D + (D / 8) * g;
#pragma unroll
                    for (int i = 0; i < MT; ++i)
                        *reinterpret_cast<float2*>(dst + 2 * i) = make_float2(o[i][hh] * inv, o[i][2 + hh] * inv);
                } else {
                    float* dst = po + ((int64_t)cur_pb + r) * D + g;
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        dst[16 * i] = o[i][hh] * inv;
                        dst[16 * i + 8] = o[i][2 + hh] * inv;
                    }
                }
                if (g == 0) plse[(int64_t)cur_pb + r] = ll > 0.f ? (mm + log2f(ll)) * kLn2 : -INFINITY;
            }
        }
    };

    bool timed_out = false;
    int nq = 0;
    for (int c = 0;; ++c) {
        const int st = c % NS;
        if (!timed_out && !mbar_wait_sleep(full + 8 * st, (c / NS) & 1)) {
            atomicOr(err, 4u);
            timed_out = true;
        }
        const uint32_t db = desc + st * 32;
        const int cp0 = ld_shared_s32(db + kDescP0), flags = ld_shared_s32(db + kDescFlags);
        if ((flags & kEnd) || timed_out) break;
        if (flags & kFirst) {
            if (have) finish_item();
            have = true;
            cm = ld_shared_s32(db + kDescCm);
            cur_pb = ld_shared_s32(db + kDescPb);
            cur_rows = ld_shared_s32(db + kDescRows);
            const int qs = ld_shared_s32(db + kDescQ);
            // Q^T fragments: row g (the N index), k-step ks -> chunks 2ks, 2ks+1
            const uint32_t qb = qbuf + qs * Lay::QSLOT;
            if constexpr (F8) {
                // row g's elements (D/4) t .. (D/4) t + D/4 - 1, in order:
                // k-step ks takes elements 4 ks .. 4 ks + 3 of the run (the
                // order of the lane's K codes below), as f16
#pragma unroll
                for (int j = 0; j < D / 32; ++j) lds128(qb + swz<D>(g, (D / 32) * t + j), qcur + 4 * j);
#pragma unroll
                for (int k = 0; k < D / 8; ++k) qcur[k] = bf16x2_to_f16x2(qcur[k]);
            } else {
#pragma unroll
                for (int kp2 = 0; kp2 < D / 32; ++kp2) {
                    const int rq = lane & 7, chunk = 4 * kp2 + (lane >> 3);
                    ldsm_x4(qb + swz<D>(rq, chunk), qcur[4 * kp2], qcur[4 * kp2 + 1], qcur[4 * kp2 + 2],
                            qcur[4 * kp2 + 3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(qempty + 8 * qs);   // the Q slot may be refilled
            ++nq;
#pragma unroll
            for (int i = 0; i < MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }
        // ---- one step of the current piece at positions cp0 .. cp0+15
        const uint32_t kb = ring + st * Lay::STAGE, vb = kb + Lay::TILEB;
        // FP8 stages go straight from the codes into MMA fragments.  The d
        // index of S^T = K Q^T is contracted, so lane (g, t) takes the D/4
        // codes (D/4) t .. of K rows g and g + 8, in order, as its k-slots
        // {2t, 2t+1, 2t+8, 2t+9} of k-steps 0, 1, ... (Q's fragments hold the
        // same elements).  In O^T = V^T P^T, d is the M index: m-tile i rows
        // g and g + 8 stand for d = (D/8) g + 2i and + 1, so the lane needs
        // the D/8 codes (D/8) g .. of V rows 2t, 2t+1, 2t+8, 2t+9 (its
        // k-slots), paired across rows with byte permutes.  The stage is
        // free as soon as the codes are in registers.
        constexpr int KWD = F8 ? D / 16 : 1, VWD = F8 ? D / 32 : 1;
        uint32_t kw[2][KWD], vw[4][VWD];
        if constexpr (F8) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int j = 0; j < D / 64; ++j) lds128(kb + fswz<D>(g + 8 * h, (D / 64) * t + j), kw[h] + 4 * j);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 2 * t + (e & 1) + 8 * (e >> 1);
                if constexpr (D == 128)
                    lds128(vb + fswz<D>(r, g), vw[e]);
                else
                    lds64(vb + fswz<D>(r, g >> 1) + 8 * (g & 1), vw[e]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + 8 * st);   // the stage may be refilled
        }
        // two accumulators halve the dependent MMA chain
        float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t ka[4];
            if constexpr (F8) {
                e4m3x4_to_f16(kw[0][ks], ka[0], ka[2]);
                e4m3x4_to_f16(kw[1][ks], ka[1], ka[3]);
                mma16816_f16((ks & 1) ? s2 : s, ka, qcur[2 * ks], qcur[2 * ks + 1]);
            } else {
                const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
                ldsm_x4(kb + swz<D>(row, 2 * ks + (lane >> 4)), ka[0], ka[1], ka[2], ka[3]);
                mma16816((ks & 1) ? s2 : s, ka, qcur[2 * ks], qcur[2 * ks + 1]);
            }
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
        const uint32_t pb0 = movtrans(F8 ? pack_f16(p00, p01) : pack_bf16(p00, p01));
        const uint32_t pb1 = movtrans(F8 ? pack_f16(p10, p11) : pack_bf16(p10, p11));
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            uint32_t va[4];
            if constexpr (F8) {
                // bytes 2 (i & 1), + 1 of word i / 2 of rows (2t, 2t+1) and (2t+8, 2t+9)
                const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
                e4m3x4_to_f16(prmt(vw[0][i / 2], vw[1][i / 2], sel), va[0], va[1]);
                e4m3x4_to_f16(prmt(vw[2][i / 2], vw[3][i / 2], sel), va[2], va[3]);
                mma16816_f16(o[i], va, pb0, pb1);
            } else {
                const int row = (lane & 7) + (lane >> 4) * 8;
                ldsm_x4_t(vb + swz<D>(row, 2 * i + ((lane >> 3) & 1)), va[0], va[1], va[2], va[3]);
                mma16816(o[i], va, pb0, pb1);
            }
        }
        __syncwarp();
        if (!F8 && lane == 0) mbar_arrive(empty + 8 * st);   // the stage may be refilled
    }
    if (have) finish_item();
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

template <int D, bool F8>
__global__ void __maxnreg__(128) decode_fused_kernel(const __grid_constant__ FusedArgs f,
                                                     const __grid_constant__ CUtensorMap tmk,
                                                     const __grid_constant__ CUtensorMap tmv) {
    using Lay = FusedLayout<D, F8>;
    using TC = DecCfg<D, F8>;
    using TL = typename TC::Lay;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Launched as a programmatic dependent of the previous kernel in the
    // stream.  Until the dependency wait below, the CTA touches only shared
    // memory, TMEM and the plan tables (uploaded from the host before the
    // previous kernel, never written by a kernel), so the set-up overlaps
    // that kernel's tail.
    const int w0 = __ldg(f.wptr + blockIdx.x), w1 = __ldg(f.wptr + blockIdx.x + 1);
    const bool tiles = w1 > w0;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + TL::OFF_TMEM);
    int* info = reinterpret_cast<int*>(sm + TL::OFF_INFO);
    const uint32_t sbar = smem_u32(sm + Lay::OFF_SBAR);
    auto full_of = [&](int c) { return sbar + (uint32_t)(c * (2 * kNSF + 2)) * 8; };
    auto empty_of = [&](int c) { return sbar + (uint32_t)(c * (2 * kNSF + 2) + kNSF) * 8; };
    auto qempty_of = [&](int c) { return sbar + (uint32_t)(c * (2 * kNSF + 2) + 2 * kNSF) * 8; };
    if (tid == 0) {
        if (tiles) tc_init_barriers<TC>(smem_u32(sm + TL::OFF_BAR));
        for (int c = 0; c < kConsumers; ++c) {
            for (int s = 0; s < kNSF; ++s) {
                mbar_init(full_of(c) + 8 * s, 33);    // the producer's 32 lanes + its descriptor release
                mbar_init(empty_of(c) + 8 * s, 1);    // the consumer
            }
            mbar_init(qempty_of(c), 1);
            mbar_init(qempty_of(c) + 8, 1);
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
    // the first records this CTA reads (plan tables) into L1 while waiting
    if (tiles && tid == 0) prefetch_l1(f.t.items + w0);
    if (!tiles && warp >= kFirstProducer && warp < kFirstConsumer && lane == 0) {
        const int gw = ((int)blockIdx.x - f.n_tile_ctas) * kConsumers + (warp - kFirstProducer);
        if (gw >= 0 && gw < f.n_init) prefetch_l1(f.narrow + gw);
    }
    // everything the previous kernel wrote is visible after this wait; the
    // merge launch may be scheduled from now on (it waits for this grid)
    grid_dep_wait();
    grid_dep_launch();

    constexpr int kStreamGate = 3;   // named barrier: tile roles done -> streaming may start
    constexpr int kTileWarps = TC::kThreads / 32;   // softmax, MMA, gather team (incl. the producers)
    if (tiles && warp < kTileWarps) {
        // the tile roles; the producer warps are part of the gather team and
        // go on to stream once the CTA's tiles are done
        const uint32_t tbase = *tslot;
        TcState st{0u, 0u, false};
        for (int w = w0; w < w1; ++w) {
            if (tid == 0) dec_tile_info(f.t, w, info);
            named_bar(kTileBar, TC::kThreads);
            const TileInfo ti{info[0], info[1], info[2], info[3], {info[4], 0}, {info[5], 0}, {info[6], 0}, INT_MAX, 0};
            tc_tile_run<TC>(f.t, &tmk, &tmv, nullptr, nullptr, ti, sm, tbase, st, tid);
            named_bar(kTileBar, TC::kThreads);
        }
        // the streaming areas overlap the tile roles' barriers
        if (tid == 0) tc_inval_barriers<TC>(smem_u32(sm + TL::OFF_BAR));
        asm volatile("bar.arrive %0, %1;\n" ::"r"(kStreamGate), "r"(kFusedThreads) : "memory");
    }
    // streaming warps of CTAs with tiles start once the tiles are done
    if (tiles && warp >= kTileWarps) named_bar(kStreamGate, kFusedThreads);
    if (warp >= kFirstProducer && warp < kFirstConsumer) {
        const int c = warp - kFirstProducer;
        const int gws = (int)blockIdx.x >= f.n_tile_ctas ? ((int)blockIdx.x - f.n_tile_ctas) * kConsumers + c : -1;
        const uint32_t sring = smem_u32(sm + Lay::OFF_SLOT + c * Lay::SLOTW);
        const uint32_t desc = smem_u32(sm + Lay::OFF_DESC + c * kNSF * 32);
        const uint32_t qb = smem_u32(sm + Lay::OFF_Q + c * 2 * Lay::QSLOT);
        if (tiles)
            stream_producer<D, kNS, F8>(f, gws, smem_u32(sm + Lay::OFF_RING + c * Lay::RING), sring, desc, qb,
                                        full_of(c), empty_of(c), qempty_of(c), lane);
        else
            stream_producer<D, kNSF, F8>(f, gws, smem_u32(sm + c * Lay::RING_F), sring, desc, qb, full_of(c),
                                         empty_of(c), qempty_of(c), lane);
    } else if (warp >= kFirstConsumer) {
        const int c = warp - kFirstConsumer;
        const uint32_t desc = smem_u32(sm + Lay::OFF_DESC + c * kNSF * 32);
        const uint32_t qb = smem_u32(sm + Lay::OFF_Q + c * 2 * Lay::QSLOT);
        if (tiles)
            stream_consumer<D, kNS, F8>(f, smem_u32(sm + Lay::OFF_RING + c * Lay::RING), desc, qb, full_of(c),
                                        empty_of(c), qempty_of(c), lane);
        else
            stream_consumer<D, kNSF, F8>(f, smem_u32(sm + c * Lay::RING_F), desc, qb, full_of(c), empty_of(c),
                                         qempty_of(c), lane);
    }
    tc_fence_before();
    __syncthreads();
    if (tiles && warp == 4) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(*tslot));
    }
}

}  // namespace

template <int D, bool F8>
int launch_decode_fused(const sgl_plan* plan, const void* q, const void* kp, const void* vp, const int32_t* r2t,
                        int64_t ld, const int32_t* seq_lens, void* o, float* lse, unsigned char* ws, float scale_log2,
                        cudaStream_t s) {
    using Lay = FusedLayout<D, F8>;
    static const int attr = (int)cudaFuncSetAttribute(decode_fused_kernel<D, F8>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::TOTAL);
    if (attr) return attr;
    const sgl_attn_params& p = plan->params;
    // the tiles' TMA views of the pools (unused, and left zero, without tiles
    // or with an FP8 pool, whose tiles load the codes with plain loads)
    CUtensorMap mk{}, mv{};
    if (plan->n_wide > 0 && !F8)
        if (const int e = tc::encode_pool_maps(kp, vp, p.num_slots, p.num_kv_heads, D, &mk, &mv)) return e;
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
    f.narrow = a.items + plan->n_wide;
    f.n_narrow = plan->n_narrow;
    f.n_init = plan->n_init;
    f.n_tile_ctas = plan->n_tile_ctas;
    f.sched = reinterpret_cast<uint32_t*>(ws + plan->off_sched);
    a.k_scale = p.k_scale;
    a.v_scale = p.v_scale;
    // Both launches are programmatic dependents of the kernel before them:
    // each waits (griddepcontrol.wait) before its first memory access, so
    // only the launch and scheduling overlap the previous grid's tail.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)plan->n_ctas);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = Lay::TOTAL;
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    int e = (int)cudaLaunchKernelEx(&cfg, decode_fused_kernel<D, F8>, f, mk, mv);
    if (e) return e;
    MergeArgs m{a.po, a.plse, reinterpret_cast<const int32_t*>(ws + plan->off_mptr),
                reinterpret_cast<const int32_t*>(ws + plan->off_ment), o, lse, a.Hq, a.Hkv, a.G};
    const int n_pairs = p.batch * a.Hkv;
    cfg.gridDim = dim3((unsigned)((n_pairs * a.G + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    return (int)cudaLaunchKernelEx(&cfg, decode_merge_kernel<bf16, D>, m, n_pairs);
}

template int launch_decode_fused<64, false>(const sgl_plan*, const void*, const void*, const void*, const int32_t*,
                                            int64_t, const int32_t*, void*, float*, unsigned char*, float, cudaStream_t);
template int launch_decode_fused<128, false>(const sgl_plan*, const void*, const void*, const void*, const int32_t*,
                                             int64_t, const int32_t*, void*, float*, unsigned char*, float,
                                             cudaStream_t);
template int launch_decode_fused<64, true>(const sgl_plan*, const void*, const void*, const void*, const int32_t*,
                                           int64_t, const int32_t*, void*, float*, unsigned char*, float, cudaStream_t);
template int launch_decode_fused<128, true>(const sgl_plan*, const void*, const void*, const void*, const int32_t*,
                                            int64_t, const int32_t*, void*, float*, unsigned char*, float,
                                            cudaStream_t);

}  // namespace sgl
