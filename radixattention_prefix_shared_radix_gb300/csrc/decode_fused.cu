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
//   all warps   (CTAs with wide items, first) the tcgen05 tile roles of
//               tc_tile.cuh over this CTA's wide items: a chunk of a shared
//               segment against up to 128 query rows (member request x query
//               head of one KV head): warps 0-3 softmax, 4 MMA, 5-14 the
//               gather team;
//   warp 2      the streaming lookup warp: pieces, slots, piece fields;
//   warps 3-6   the streaming producers (bulk copies of whole token rows);
//   warps 7-14  streaming consumers, 8 query rows of one KV head each
//   (in CTAs with wide items, the streaming roles start once the tiles are
//   done).
// A narrow piece is a run of positions of one request segment (a request's
// own suffix, or a small group's) for a block of up to 8 consecutive KV
// heads with at most 8 query rows per head (members x G query heads), or of
// up to 4 heads with at most 16 rows per head (two consumer warps each).  In
// the pool [slot, Hkv, d] a token's K (or V) row for those heads is one
// contiguous run of nh * d elements, moved with one cp.async.bulk.
// Measured on GB300: random 2 KB token rows gather at 6.8-7.1 TB/s from 152
// SMs; on 32 SMs (HBM not saturated) one warp issuing them reaches 54 GB/s
// per SM and four warps 117 GB/s (a warp gets about one bulk copy through
// every 100 cycles), hence four producer warps; 256-byte rows of one head,
// as 16-byte cp.async, stalled near 32 GB/s per SM on the copy issue.  The
// lookup warp takes every global-latency wait (piece counter, records,
// slot table) off the producers.  The tiles are bound by latency and the tensor
// pipe, the streams by HBM.  The planner puts the wide items on the first
// CTAs (as many as balance the streaming work); their streaming warps wait
// at a barrier until the tiles are done and then take pieces from the
// run-time counter, so an SM never runs both kinds at once (measured:
// co-running them cost the streams most of their instruction-cache hits).
//
// Streaming ring: NSF stages of 16 positions, each the 16 K rows then the
// 16 V rows of those positions, a row every nh * d * (element bytes) + 16
// bytes: the 16-byte pad puts 8 consecutive rows in distinct banks, so the
// consumers' ldmatrix reads need no swizzle (a bulk copy lands a whole row
// contiguously).  Per stage a FULL mbarrier (the producer's arrival with the
// stage's byte count; the copies complete it), an EMPTY mbarrier (one
// arrival per consumer warp) and a 64-byte descriptor (first position,
// flags; for a piece's first step the piece's fields and member requests).
// The lookup warp fills a slot ring of 8 steps (4-byte cp.async of each
// step's slots, plus the piece fields), so no producer register ever waits
// on a load in flight.  At a piece's first step each consumer lane loads its
// query row's fragment straight from q (L2-resident: q is read by every
// piece of its requests); nothing in the ring waits for the consumers to be
// done with the previous piece, so the next piece's copies are in flight
// while they finish it (measured: a Q slot refilled between pieces left the
// ring empty for ~2 us at every piece boundary).
//
// Consumer warp, per 16-position step, for its KV head and 8 query rows of
// the piece (mma.sync m16n8k16, bf16 in, fp32 acc; the query rows in the
// MMA's N dimension):
//   S^T [16 pos x 8 rows] = K [16 x d] . Q^T [d x 8 rows]
//   O^T [d x 8 rows]     += V^T [d x 16 pos] . P^T [16 pos x 8 rows]
// ldmatrix for K, ldmatrix.trans for V^T; P^T moves from the accumulator
// layout to the B-operand layout with movmatrix.  Apart from a piece's
// query fragments, the consumers' loop touches nothing but shared memory.
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

constexpr int kHB = kDecHeadBlock;                       // consumer warps = KV heads of a piece (at most)
constexpr int kNP = 16;                                  // KV positions per step
constexpr int kSQ = 8;                                   // slot ring entries (lookups ahead of the copies)
constexpr int kSlotEntry = 128;                          // 16 slots + step and piece fields (see below)
constexpr int kLookup = 2;                               // the lookup warp
constexpr int kFirstProducer = 3;
constexpr int kProducers = 4;                            // each issues 8 of a stage's 32 row copies
constexpr int kFirstConsumer = kFirstProducer + kProducers;
constexpr int kFusedThreads = 32 * (kFirstConsumer + kHB);
static_assert(DecCfg<128>::kThreads == kFusedThreads && DecCfg<64>::kThreads == kFusedThreads,
              "the tile roles take the whole CTA");
static_assert((kSQ & (kSQ - 1)) == 0, "slot ring");
static_assert((2 * kNP) % kProducers == 0 && 2 * kNP / kProducers <= 32, "row copies per producer warp");

template <int D, bool F8 = false>
struct FusedLayout {
    using TL = typename DecCfg<D, F8>::Lay;
    static constexpr int ES = F8 ? 1 : 2;                // bytes per pool element
    static constexpr int PITCH = kHB * D * ES + 16;      // one token's K (or V) row of a head block, padded
    static constexpr int STAGE = 2 * kNP * PITCH;        // K rows, then V rows
    static constexpr int SLOTW = kSQ * kSlotEntry;
    static constexpr int DESC = 64;                      // stage descriptor bytes
    static constexpr int FIXED = 1024 + SLOTW + 8 * DESC + 64 + (2 * 8 + 2 * kSQ) * 8 + 1024;
    static constexpr int NSF0 = (232448 - FIXED) / STAGE;
    static constexpr int NSF = NSF0 > 8 ? 8 : NSF0;      // ring stages
    // Layout: the tile roles' TMEM address and broadcast area (up to
    // TL::KEEP); from 1024 the ring, the slot ring and the stage
    // descriptors.  These are used only once the CTA's tiles are done, so
    // they overlap the rest of the tile roles' area (TL::KEEP .. TL::END:
    // stages, barriers, staging).  The streaming barriers, initialised at
    // launch, come after everything.
    static constexpr int OFF_RING = 1024;
    static constexpr int OFF_SLOT = OFF_RING + NSF * STAGE;
    static constexpr int OFF_DESC = OFF_SLOT + SLOTW;
    static constexpr int OFF_LREC = OFF_DESC + NSF * DESC;   // launch piece: record (32 B), members (32 B)
    static constexpr int END_S = OFF_LREC + 64;
    // FULL[NSF], EMPTY[NSF], SLOTFULL[kSQ], SLOTFREE[kSQ]
    static constexpr int OFF_SBAR = ((END_S > TL::END ? END_S : TL::END) + 7) / 8 * 8;
    static constexpr int END = OFF_SBAR + (2 * NSF + 2 * kSQ) * 8;
    static constexpr int TOTAL = END + 1024;             // + alignment slack
    static_assert(NSF >= 3, "ring depth");
    static_assert(OFF_SBAR >= TL::END && OFF_SBAR >= END_S, "streaming barriers clear of every other area");
    static_assert(TOTAL <= 232448, "shared memory per CTA");
    static_assert(TL::KEEP <= OFF_RING, "the ring clears the tile roles' kept area");
};

struct FusedArgs {
    TcArgs t;
    const int32_t* wptr;   // [n_ctas + 1] wide items of each CTA
    const DecItem* narrow; // narrow pieces, longest first
    int n_narrow;
    int n_init;            // pieces assigned at launch: streaming CTA w starts on piece w
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
constexpr int kFirst = 1;   // first step of its piece: the descriptor carries the piece's fields
constexpr int kEnd = 4;     // no more pieces: the consumers stop

// slot-ring entry (one looked-up step): 16 slots, then
constexpr int kEntKvh = 64, kEntP0 = 68, kEntFlags = 72, kEntCm = 76, kEntPb = 80, kEntNh = 84, kEntNm = 88;
constexpr int kEntMem = 96;   // kDecPieceMembers ints: the piece's member requests (first step only)
static_assert(kEntMem + 4 * kDecPieceMembers <= kSlotEntry, "a slot entry holds a piece's members");
// stage descriptor (a piece's first step also carries the piece's first KV
// head and member requests, from which the consumers load their query rows)
constexpr int kDescP0 = 0, kDescFlags = 4, kDescCm = 8, kDescPb = 12, kDescRows = 16, kDescNh = 20, kDescKvh = 24;
constexpr int kDescMem = 32;   // kDecPieceMembers ints

// ---------------------------------------------------------------------------
// Lookup warp (one per CTA)
// ---------------------------------------------------------------------------
// Walks this CTA's pieces (its launch piece, whose record and members were
// loaded before the dependency wait, then pieces taken from the run-time
// counter) and fills the slot ring up to kSQ steps ahead of the producers:
// per step the 16 slots (4-byte cp.async from req_to_token; positions past
// the piece's end marked), the step's first KV head, position and flags,
// and for a piece's first step its partial base, clamped end, head and
// member counts and member requests.  Each entry's barrier (SLOTFULL)
// completes when the lanes' cp.async have landed and lane 0 has written the
// fields; the producers free it (SLOTFREE).  An entry with no KV head ends
// the stream.  Global loads (the counter, records, seq_lens) stall only this
// warp, which runs ahead of the copies.
template <int D, bool F8>
__device__ __noinline__ void stream_lookup(const FusedArgs& f, int gw, uint32_t lrec, uint32_t sring,
                                           uint32_t sfull, uint32_t sfree, int lane) {
    constexpr int32_t kPastEnd = INT32_MIN;
    const int32_t* const r2t = f.t.r2t;
    const int32_t* const members = f.t.members;
    const int32_t* const seq_lens = f.t.seq_lens;
    const int64_t ld = f.t.ld;
    uint32_t* const err = f.t.err;
    const DecItem* const pieces = f.narrow;
    const int n_narrow = f.n_narrow;
    uint32_t* const sched = f.sched;
    const bool launch = gw >= 0 && gw < f.n_init;
    bool timed_out = false;
    int nlook = 0;
    // one ring entry: wait for it to be free, fill it, arm its barrier.  A
    // piece's first entry also records its end clamped to seq_len (len, whose
    // load is only waited for once the slot lookups are issued)
    auto entry = [&](int kvh, int row, int p0, int e, int flags, int len, int pb, int nh, int nm, int mem) {
        const int ent = nlook & (kSQ - 1);
        const uint32_t eb = sring + ent * kSlotEntry;
        if (!timed_out && !mbar_wait(sfree + 8 * ent, ((nlook / kSQ) & 1) ^ 1)) {
            atomicOr(err, 4u);
            timed_out = true;
        }
        if (timed_out) return;
        if (lane < kNP) {
            const int p = p0 + lane;
            if (kvh >= 0 && p < e)
                cp_async4(eb + lane * 4, r2t + (int64_t)row * ld + p);
            else
                st_shared_s32(eb + lane * 4, kPastEnd);
        }
        if (lane == 0) {
            st_shared_s32(eb + kEntKvh, kvh);
            st_shared_s32(eb + kEntP0, p0);
            st_shared_s32(eb + kEntFlags, flags);
            if (flags & kFirst) {
                int cm = e;
                if (e > len) {   // planned beyond seq_len: mask the excess, flag it
                    atomicOr(err, 2u);
                    cm = len > p0 ? len : p0;
                }
                st_shared_s32(eb + kEntCm, cm);
                st_shared_s32(eb + kEntPb, pb);
                st_shared_s32(eb + kEntNh, nh);
                st_shared_s32(eb + kEntNm, nm);
            }
        }
        if ((flags & kFirst) && lane < kDecPieceMembers) st_shared_s32(eb + kEntMem + 4 * lane, mem);
        cp_async_arrive_noinc(sfull + 8 * ent);   // each lane, once its lookups have landed
        __syncwarp();
        if (lane == 0) mbar_arrive(sfull + 8 * ent);   // the fields
        ++nlook;
    };
    bool first_piece = true;
    for (;;) {
        int row, b, e, kvh, mb, nm, pb, nh, mem;
        if (first_piece && launch) {
            row = ld_shared_s32(lrec); b = ld_shared_s32(lrec + 4); e = ld_shared_s32(lrec + 8);
            kvh = ld_shared_s32(lrec + 12); mb = ld_shared_s32(lrec + 16); nm = ld_shared_s32(lrec + 20);
            pb = ld_shared_s32(lrec + 24); nh = ld_shared_s32(lrec + 28);
            mem = lane < kDecPieceMembers ? ld_shared_s32(lrec + 32 + 4 * lane) : 0;
        } else {
            int taken = 0;
            if (lane == 0) taken = (int)atomicAdd(sched, 1u);
            taken = __shfl_sync(0xffffffffu, taken, 0);
            if (taken >= n_narrow) break;
            const int4* rp = reinterpret_cast<const int4*>(pieces + taken);
            const int4 x = __ldg(rp), y = __ldg(rp + 1);
            row = x.x; b = x.y; e = x.z; kvh = x.w;
            mb = y.x; nm = y.y; pb = y.z; nh = y.w;
            mem = lane < nm ? __ldg(members + mb + lane) : 0;
        }
        first_piece = false;
        int len = __ldg(seq_lens + row);
        if (e == kDecToSeqEnd) {
            // a request's trailing piece runs to its length now (within its
            // row of the table; a length below the piece's start is an error)
            if (len > ld || len < b) {
                if (lane == 0) atomicOr(err, 2u);
                len = len > ld ? (int)ld : b;
            }
            e = len;
        }
        // at least one step, so that an empty piece still writes its
        // (empty) partial rows for the merge
        for (int sp = b; sp < e || sp == b; sp += kNP)
            entry(kvh, row, sp, e, sp == b ? kFirst : 0, len, pb, nh, nm, mem);
    }
    entry(-1, 0, 0, 0, 0, 0, 0, 0, 0, 0);   // the end of the stream
    cp_async_wait<0>();
    // The last lookup warp to finish restores the counter for the next call
    // (every CTA has taken its last number by then).
    if (lane == 0) {
        if (atomicAdd(sched + 1, 1u) + 1 == gridDim.x) {
            sched[0] = (uint32_t)f.n_init;
            sched[1] = 0u;
            __threadfence();
        }
    }
}

// ---------------------------------------------------------------------------
// Producer warp p of kProducers
// ---------------------------------------------------------------------------
// For each step (slot-ring entry, in order): waits for the entry and for the
// ring stage to be free, zero-fills its rows without data (positions past
// the piece's end, or slots outside the pool), arrives on the stage's FULL
// barrier with its byte count and issues its bulk copies: lane t < 8 moves
// row 8p + t of the stage (rows 0-15 the K rows of the step's 16 positions,
// 16-31 the V rows).  Measured on GB300: one warp gets a bulk copy through
// about every 100 cycles, so four warps share the stage's 32 row copies.
// Producer 0 also writes the stage descriptor (for a piece's first step
// with the piece's fields and member requests).  A piece's first step waits
// for nothing but a free stage, so the next piece's data is in flight while
// the consumers finish the last one.  The entry is freed once read.
template <int D, bool F8>
__device__ __noinline__ void stream_producer(const FusedArgs& f, int pw, uint32_t ring, uint32_t sring,
                                             uint32_t desc, uint32_t full, uint32_t empty, uint32_t sfull,
                                             uint32_t sfree, int lane) {
    using Lay = FusedLayout<D, F8>;
    constexpr int NS = Lay::NSF;
    constexpr int ES = Lay::ES;
    constexpr int32_t kPastEnd = INT32_MIN;
    constexpr int RPW = 2 * kNP / kProducers;   // rows per producer warp and step
    // argument fields in registers: every asm below clobbers memory
    const uint8_t* const kp = reinterpret_cast<const uint8_t*>(f.t.kp);
    const uint8_t* const vp = reinterpret_cast<const uint8_t*>(f.t.vp);
    uint32_t* const err = f.t.err;
    const int Hkv = f.t.Hkv, G = f.t.G;
    const int64_t num_slots = f.t.num_slots;
    // streamed K/V rows are read once: evict them from L2 first, which keeps
    // the code, the tables and the partial rows there across calls
    const uint64_t kv_pol = l2_evict_first_policy();
    const bool lead = pw == 0;
    const int idx = pw * RPW + lane;          // this lane's row of a stage (lane < RPW)
    const bool mine = lane < RPW;
    const int tok = idx & (kNP - 1);

    // After a wait gives up, the producer stops touching the ring and its
    // barriers (the consumers' and the lookup warp's own bounded waits end
    // their loops).
    bool timed_out = false;
    int cur_nh = 0;        // KV heads of the piece being issued
    int last_armed = -1;   // last step whose FULL phase this warp's copies complete
    int last_arrived = -1; // last step that arrived on a FULL barrier (armed, or the end marker)
    for (int r = 0; !timed_out; ++r) {
        const int ent = r & (kSQ - 1);
        const uint32_t eb = sring + ent * kSlotEntry;
        if (!mbar_wait(sfull + 8 * ent, (uint32_t)(r / kSQ) & 1u)) {
            atomicOr(err, 4u);
            timed_out = true;
            break;
        }
        const int kvh = ld_shared_s32(eb + kEntKvh);
        const int flags = ld_shared_s32(eb + kEntFlags);
        const int st = r % NS;
        if (!mbar_wait(empty + 8 * st, ((r / NS) & 1) ^ 1)) {
            atomicOr(err, 4u);
            timed_out = true;
            break;
        }
        const uint32_t db = desc + st * Lay::DESC;
        const uint32_t fb = full + 8 * st;
        const uint32_t sb = ring + st * Lay::STAGE;
        if (kvh < 0) {
            if (lane == 0) {
                if (lead) st_shared_s32(db + kDescFlags, kEnd);
                mbar_arrive(fb);
            }
            last_arrived = r;
            __syncwarp();
            if (lane == 0) mbar_arrive(sfree + 8 * ent);
            break;
        }
        const bool first = (flags & kFirst) != 0;
        if (first) cur_nh = ld_shared_s32(eb + kEntNh);
        const uint32_t rowb = (uint32_t)(cur_nh * D * ES);
        int32_t sl = mine ? ld_shared_s32(eb + tok * 4) : kPastEnd;
        bool ok = mine && sl != kPastEnd;
        if (ok && (sl < 0 || sl >= num_slots)) {
            if (idx < kNP) atomicOr(err, 1u);
            ok = false;
        }
        const uint32_t vmask = __ballot_sync(0xffffffffu, ok);
        // rows without data are zeroed: their scores are masked, and a zero V
        // row keeps 0 * V finite
        uint32_t zm = ~vmask & ((1u << RPW) - 1u);
        if (zm) {
            while (zm) {
                const int b = __ffs(zm) - 1;
                zm &= zm - 1;
                const int zi = pw * RPW + b;
                const uint32_t zr = sb + (uint32_t)((zi >> 4) * kNP + (zi & (kNP - 1))) * Lay::PITCH;
                for (uint32_t c = (uint32_t)lane * 16u; c < rowb; c += 512u) st_shared_v4(zr + c, 0u, 0u, 0u, 0u);
            }
            // the stage's next use writes these rows through the async proxy
            fence_proxy_async_smem();
        }
        const uint32_t bytes = (uint32_t)__popc(vmask) * rowb;
        if (lead && lane == 0) {
            st_shared_s32(db + kDescP0, ld_shared_s32(eb + kEntP0));
            st_shared_s32(db + kDescFlags, flags);
            if (first) {
                st_shared_s32(db + kDescCm, ld_shared_s32(eb + kEntCm));
                st_shared_s32(db + kDescPb, ld_shared_s32(eb + kEntPb));
                st_shared_s32(db + kDescRows, ld_shared_s32(eb + kEntNm) * G);
                st_shared_s32(db + kDescNh, cur_nh);
                st_shared_s32(db + kDescKvh, kvh);
            }
        }
        if (lead && first && lane < kDecPieceMembers)
            st_shared_s32(db + kDescMem + 4 * lane, ld_shared_s32(eb + kEntMem + 4 * lane));
        __syncwarp();
        if (lane == 0) mbar_expect_tx(fb, bytes);   // the arrival, plus the bytes the copies complete
        __syncwarp();
        if (ok)
            bulk_g2s_pol(sb + (uint32_t)((idx >> 4) * kNP + tok) * Lay::PITCH,
                         (idx < kNP ? kp : vp) + ((int64_t)sl * Hkv + kvh) * (D * ES), rowb, fb, kv_pol);
        last_armed = last_arrived = r;
        __syncwarp();   // every lane has read the entry
        if (lane == 0) mbar_arrive(sfree + 8 * ent);
    }
    // This warp's bulk copies have landed before it leaves (normally long
    // since: the consumers read them): an armed phase completes only when
    // they have.  Only steps whose stage no later step arrived on are waited
    // for (a later phase of the same stage would flip the parity back).
    // Bounded waits.
    const int s0 = last_arrived - NS + 1 > 0 ? last_arrived - NS + 1 : 0;
    for (int s = s0; s <= last_armed; ++s)
        if (!mbar_wait(full + 8 * (s % NS), (uint32_t)(s / NS) & 1u)) atomicOr(err, 4u);
}

// ---------------------------------------------------------------------------
// Consumer warp c: 8 query rows of one KV head of each piece (idle, but
// keeping the barrier counts, when the piece has fewer heads or rows); only
// shared memory in its loop (stages, descriptors) but for a piece's query
// fragments
// ---------------------------------------------------------------------------
template <int D, bool F8>
__device__ __noinline__ void stream_consumer(const FusedArgs& f, int c, uint32_t ring, uint32_t desc, uint32_t full,
                                             uint32_t empty, int lane) {
    using Lay = FusedLayout<D, F8>;
    constexpr int NS = Lay::NSF;
    constexpr int P = Lay::PITCH;
    constexpr int MT = D / 16;                 // m-tiles of O^T
    const int g = lane >> 2, t = lane & 3;
    float* const po = f.t.po;
    float* const plse = f.t.plse;
    uint32_t* const err = f.t.err;
    const int G = f.t.G;
    // FP8 pools: the K scale goes into the score scale, the V scale into the
    // final normalisation (both are per tensor, so they factor out)
    const float sc = F8 ? f.t.scale_log2 * f.t.k_scale : f.t.scale_log2;
    const float vsc = F8 ? f.t.v_scale : 1.f;
    // Per piece: a head with at most 8 query rows takes one consumer warp
    // (warp c: KV head kvh + c), one with more takes two (warp c: head
    // kvh + c / 2, rows 8 (c % 2) ..); hw is this warp's head in the piece,
    // r0 its first row of the head.
    uint32_t hoff = 0;   // this warp's head within a K/V row
    int hw = 0, r0 = 0;
    const bf16* const qp = f.t.q;
    const int Hq = f.t.Hq;

    uint32_t qcur[D / 8];
    float o[MT][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool have = false, active = false;
    int cur_pb = 0, cur_rows = 0, cur_nh = 0, cm = 0;
    auto finish_item = [&]() {
        float s0 = l0, s1 = l1;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, off);
            s1 += __shfl_xor_sync(0xffffffffu, s1, off);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = r0 + 2 * t + hh;   // query row of this head: member r / G, query head r % G
            if (r < cur_rows) {
                const int64_t prow = (int64_t)cur_pb + ((r / G) * cur_nh + hw) * G + r % G;
                const float ll = hh ? s1 : s0, mm = hh ? m1 : m0;
                const float inv = ll > 0.f ? vsc / ll : 0.f;
                if constexpr (F8) {
                    // m-tile i rows g, g + 8 stand for d = (D/8) g + 2i, + 1
                    float* dst = po + prow * D + (D / 8) * g;
#pragma unroll
                    for (int i = 0; i < MT; ++i)
                        *reinterpret_cast<float2*>(dst + 2 * i) = make_float2(o[i][hh] * inv, o[i][2 + hh] * inv);
                } else {
                    float* dst = po + prow * D + g;
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        dst[16 * i] = o[i][hh] * inv;
                        dst[16 * i + 8] = o[i][2 + hh] * inv;
                    }
                }
                if (g == 0) plse[prow] = ll > 0.f ? (mm + log2f(ll)) * kLn2 : -INFINITY;
            }
        }
    };

    for (int cs = 0;; ++cs) {
        const int st = cs % NS;
        if (!mbar_wait(full + 8 * st, (cs / NS) & 1)) {
            atomicOr(err, 4u);
            break;
        }
        const uint32_t db = desc + st * Lay::DESC;
        const int cp0 = ld_shared_s32(db + kDescP0), flags = ld_shared_s32(db + kDescFlags);
        if (flags & kEnd) break;
        if (flags & kFirst) {
            if (have && active) finish_item();
            have = true;
            cm = ld_shared_s32(db + kDescCm);
            cur_pb = ld_shared_s32(db + kDescPb);
            cur_rows = ld_shared_s32(db + kDescRows);
            cur_nh = ld_shared_s32(db + kDescNh);
            const int wph = cur_rows > 8 ? 2 : 1;   // consumer warps per head
            hw = c / wph;
            r0 = (c - hw * wph) * 8;
            active = hw < cur_nh && r0 < cur_rows;
            hoff = (uint32_t)(hw * D * Lay::ES);
            if (active) {
                // this lane's query row r0 + g: member (r0 + g) / G of the
                // piece, query head (kvh + hw) G + (r0 + g) % G; zero past the
                // piece's rows (their output columns are never used)
                const int rq = r0 + g;
                const bool okq = rq < cur_rows;
                const int mq = okq ? ld_shared_s32(db + kDescMem + 4 * (rq / G)) : 0;
                const bf16* qrow =
                    qp + ((int64_t)mq * Hq + (ld_shared_s32(db + kDescKvh) + hw) * G + rq % G) * D;
                // Q^T fragments: row g (the N index), k-step ks -> chunks 2ks, 2ks+1
                if constexpr (F8) {
                    // row g's elements (D/4) t .. (D/4) t + D/4 - 1, in order:
                    // k-step ks takes elements 4 ks .. 4 ks + 3 of the run (the
                    // order of the lane's K codes below), as f16
                    const uint4* src = reinterpret_cast<const uint4*>(qrow + (D / 4) * t);
#pragma unroll
                    for (int j = 0; j < D / 32; ++j) {
                        const uint4 v = okq ? __ldg(src + j) : make_uint4(0u, 0u, 0u, 0u);
                        qcur[4 * j] = v.x;
                        qcur[4 * j + 1] = v.y;
                        qcur[4 * j + 2] = v.z;
                        qcur[4 * j + 3] = v.w;
                    }
                    uint32_t bad = 0u;
#pragma unroll
                    for (int k = 0; k < D / 8; ++k) qcur[k] = bf16x2_to_f16x2_chk(qcur[k], bad);
                    if (bad) atomicOr(f.t.err, kErrQRange);
                } else {
                    // chunk k (elements 8k .. 8k+7): the lane's pair 2t, 2t+1
                    const uint32_t* src = reinterpret_cast<const uint32_t*>(qrow) + t;
#pragma unroll
                    for (int k = 0; k < D / 8; ++k) qcur[k] = okq ? __ldg(src + 4 * k) : 0u;
                }
            }
#pragma unroll
            for (int i = 0; i < MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }
        if (!active) {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + 8 * st);
            continue;
        }
        // ---- one step of the current piece at positions cp0 .. cp0+15
        const uint32_t kb = ring + st * Lay::STAGE + hoff, vb = kb + kNP * P;
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
                for (int j = 0; j < D / 64; ++j) lds128(kb + (g + 8 * h) * P + ((D / 64) * t + j) * 16, kw[h] + 4 * j);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 2 * t + (e & 1) + 8 * (e >> 1);
                if constexpr (D == 128)
                    lds128(vb + r * P + 16 * g, vw[e]);
                else
                    lds64(vb + r * P + 8 * g, vw[e]);
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
                ldsm_x4(kb + row * P + (2 * ks + (lane >> 4)) * 16, ka[0], ka[1], ka[2], ka[3]);
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
                ldsm_x4_t(vb + row * P + (2 * i + ((lane >> 3) & 1)) * 16, va[0], va[1], va[2], va[3]);
                mma16816(o[i], va, pb0, pb1);
            }
        }
        if constexpr (!F8) {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + 8 * st);   // the stage may be refilled
        }
    }
    if (have && active) finish_item();
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
    constexpr int NSF = Lay::NSF;
    const uint32_t sbar = smem_u32(sm + Lay::OFF_SBAR);
    const uint32_t sfull = sbar, sempty = sbar + 8 * NSF;
    const uint32_t slfull = sbar + 16 * NSF, slfree = slfull + 8 * kSQ;
    if (tid == 0) {
        if (tiles) tc_init_barriers<TC>(smem_u32(sm + TL::OFF_BAR));
        for (int s = 0; s < NSF; ++s) {
            mbar_init(sfull + 8 * s, kProducers);   // every producer's arrival (with its bytes)
            mbar_init(sempty + 8 * s, kHB);         // every consumer warp
        }
        for (int e = 0; e < kSQ; ++e) {
            mbar_init(slfull + 8 * e, 33);          // the lookup lanes' cp.async + the fields
            mbar_init(slfree + 8 * e, kProducers);  // every producer
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
    // a streaming CTA's launch piece: its record and members (plan tables)
    // into shared memory while the previous kernel finishes
    const int gw = !tiles && (int)blockIdx.x >= f.n_tile_ctas ? (int)blockIdx.x - f.n_tile_ctas : -1;
    const uint32_t lrec = smem_u32(sm + Lay::OFF_LREC);
    if (warp == kLookup && gw >= 0 && gw < f.n_init) {
        const int4* rp = reinterpret_cast<const int4*>(f.narrow + gw);
        const int4 x = __ldg(rp), y = __ldg(rp + 1);
        if (lane == 0) {
            st_shared_v4(lrec, (uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w);
            st_shared_v4(lrec + 16, (uint32_t)y.x, (uint32_t)y.y, (uint32_t)y.z, (uint32_t)y.w);
        }
        if (lane < kDecPieceMembers)
            st_shared_s32(lrec + 32 + 4 * lane, lane < y.y ? __ldg(f.t.members + y.x + lane) : 0);
        __syncwarp();
    }
    // everything the previous kernel wrote is visible after this wait; the
    // merge launch may be scheduled from now on (it waits for this grid)
    grid_dep_wait();
    grid_dep_launch();

    static_assert(TC::kThreads == kFusedThreads, "every warp has a tile role");
    if (tiles) {
        // the tile roles (all warps); warps 2-14 go on to stream (lookup,
        // producers, consumers) once the CTA's tiles are done
        const uint32_t tbase = *tslot;
        TcState st{0u, 0u, false};
        for (int w = w0; w < w1; ++w) {
            if (tid == 0) dec_tile_info(f.t, w, info);
            named_bar(kTileBar, TC::kThreads);
            const TileInfo ti{info[0], info[1], info[2], info[3], {info[4], 0}, {info[5], 0}, {info[6], 0}, INT_MAX, 0};
            tc_tile_run<TC>(f.t, &tmk, &tmv, nullptr, nullptr, ti, sm, tbase, st, tid);
            named_bar(kTileBar, TC::kThreads);
        }
        // the streaming areas overlap the tile roles' barriers: invalidated
        // before any streaming role starts
        if (tid == 0) tc_inval_barriers<TC>(smem_u32(sm + TL::OFF_BAR));
        named_bar(kTileBar, TC::kThreads);
    }
    const uint32_t ring = smem_u32(sm + Lay::OFF_RING);
    const uint32_t desc = smem_u32(sm + Lay::OFF_DESC);
    const uint32_t sring = smem_u32(sm + Lay::OFF_SLOT);
    if (warp == kLookup) {
        stream_lookup<D, F8>(f, gw, lrec, sring, slfull, slfree, lane);
    } else if (warp >= kFirstProducer && warp < kFirstConsumer) {
        stream_producer<D, F8>(f, warp - kFirstProducer, ring, sring, desc, sfull, sempty, slfull,
                               slfree, lane);
    } else if (warp >= kFirstConsumer) {
        stream_consumer<D, F8>(f, warp - kFirstConsumer, ring, desc, sfull, sempty, lane);
    }
    // the tiles' partial rows went out as bulk copies from the softmax
    // threads (0-127): complete before the grid is
    if (tiles && tid < 128) bulk_wait_all();
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
    cfg.gridDim = dim3((unsigned)merge_blocks<D>(n_pairs, a.G));
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
