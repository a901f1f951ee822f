// Prefix-group scheduler for decode: turns the batch's prefix groups into
// GPU work items and the per-(request, KV head) merge lists.
//
// A segment (a run of positions shared by a set of member requests, read
// from one representative row) is the unit of sharing: its K/V are read
// once for all members and all query heads of a KV head -- "computed once,
// referenced many times" ("SGLang：从前端 DSL 到 SRT 服务运行时", section
// "用基数树实现前缀复用"; bhfrc.com/news/45689 §1.3).  The pages give no
// kernel schedule; this one is ours:
//   * a segment with more than 8 query rows (member x query head of a KV
//     head; a prefix shared by many requests) becomes tensor-core tiles:
//     member blocks of up to 128 rows x chunks of whole 128-position
//     multiples, dealt to a set of tile CTAs sized with the streaming work
//     (cost model below);
//   * every other segment (at most 16 rows per KV head: a request's own
//     suffix, or a small group) is narrow: its positions, for blocks of up
//     to 8 consecutive KV heads (4 when a head has more than 8 rows; a
//     token's K or V row of those heads is one contiguous run in the pool),
//     are cut into pieces handed to the streaming CTAs at run time, longest
//     first;
//   * each item writes its rows' normalised partial O and LSE (fp32); the
//     merge list of (request, KV head) names every partial row to combine.
// The fp32 path runs the same items one CTA each.

#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "common.h"

namespace sgl {

int query_num_sms(int32_t requested) {
    if (requested > 0) return requested;
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
        return n;
    cudaGetLastError();
    return 152;
}

int check_params(const sgl_attn_params* p) {
    if (!p) return SGL_ERR_INVALID_ARG;
    if (p->batch < 0 || p->num_qo_heads <= 0 || p->num_kv_heads <= 0 || p->num_slots < 0 || p->page_size < 1)
        return SGL_ERR_INVALID_ARG;
    if (p->dtype != SGL_DTYPE_F32 && p->dtype != SGL_DTYPE_BF16 && p->dtype != SGL_DTYPE_BF16_FP8KV)
        return SGL_ERR_UNSUPPORTED;
    if (p->dtype == SGL_DTYPE_BF16_FP8KV && !(p->k_scale > 0.f && p->v_scale > 0.f)) return SGL_ERR_INVALID_ARG;
    if (p->head_dim != 64 && p->head_dim != 128) return SGL_ERR_UNSUPPORTED;
    if (p->num_qo_heads % p->num_kv_heads) return SGL_ERR_UNSUPPORTED;
    int G = p->num_qo_heads / p->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return SGL_ERR_UNSUPPORTED;
    // slot * Hkv + head is a 32-bit row coordinate of the pools' TMA view
    if (p->num_slots * p->num_kv_heads > INT32_MAX) return SGL_ERR_UNSUPPORTED;
    return SGL_OK;
}

int validate_groups(int32_t B, const int32_t* seq_lens, const sgl_prefix_groups* g) {
    const int32_t nseg = g->num_segments;
    if (nseg < 0 || (nseg > 0 && (!g->seg_begin || !g->seg_end || !g->seg_row || !g->seg_member_ptr ||
                                  !g->seg_members)))
        return SGL_ERR_INVALID_ARG;

    // Validate: every request's segments tile [0, seq_len) exactly, every
    // member holds the segment's positions, representatives are members.
    std::vector<std::vector<std::pair<int32_t, int32_t>>> cover(B);
    if (nseg > 0 && g->seg_member_ptr[0] != 0) return SGL_ERR_INVALID_ARG;
    for (int32_t s = 0; s < nseg; ++s) {
        int32_t b = g->seg_begin[s], e = g->seg_end[s], rep = g->seg_row[s];
        int32_t m0 = g->seg_member_ptr[s], m1 = g->seg_member_ptr[s + 1];
        if (b < 0 || e <= b || rep < 0 || rep >= B || m1 <= m0 || m1 > g->num_members) return SGL_ERR_INVALID_ARG;
        bool rep_is_member = false;
        for (int32_t i = m0; i < m1; ++i) {
            int32_t r = g->seg_members[i];
            if (r < 0 || r >= B || seq_lens[r] < e) return SGL_ERR_INVALID_ARG;
            if (i > m0 && r <= g->seg_members[i - 1]) return SGL_ERR_INVALID_ARG;
            rep_is_member |= (r == rep);
            cover[r].push_back({b, e});
        }
        if (!rep_is_member) return SGL_ERR_INVALID_ARG;
    }
    for (int32_t r = 0; r < B; ++r) {
        std::sort(cover[r].begin(), cover[r].end());
        int32_t at = 0;
        for (auto& iv : cover[r]) {
            if (iv.first != at) return SGL_ERR_INVALID_ARG;
            at = iv.second;
        }
        if (at != seq_lens[r]) return SGL_ERR_INVALID_ARG;
    }
    return SGL_OK;
}

}  // namespace sgl

extern "C" {

int sgl_decode_plan(const sgl_attn_params* p, const int32_t* seq_lens, const sgl_prefix_groups* g,
                    sgl_plan** plan_out, size_t* workspace_bytes) {
    int st = sgl::check_params(p);
    if (st) return st;
    if (!g || !plan_out || !workspace_bytes) return SGL_ERR_INVALID_ARG;
    const int32_t B = p->batch;
    if (B > 0 && !seq_lens) return SGL_ERR_INVALID_ARG;
    const int32_t G = p->num_qo_heads / p->num_kv_heads;
    const int32_t Hkv = p->num_kv_heads;
    const int32_t nseg = g->num_segments;
    st = sgl::validate_groups(B, seq_lens, g);
    if (st) return st;

    // Narrow segments (at most 16 query rows per KV head: members x query
    // heads of the group) go to the streaming warps; wider ones to the
    // tensor-core tiles in member blocks of up to 128 rows.
    // (a piece carries at most kDecPieceMembers member requests)
    const int32_t MBn = std::max(1, std::min(sgl::kDecPieceMembers, 16 / G));
    const int32_t MBw = std::max(1, 128 / G);
    const int sms = sgl::query_num_sms(p->num_sms);

    // Narrow work streams in blocks of consecutive KV heads (one stream per
    // CTA): up to 8 heads with one consumer warp each when a head has at
    // most 8 query rows, else up to 4 heads with two consumer warps each;
    // the fp32 kernel runs one item per CTA and takes one head per item.
    auto head_block = [&](int32_t nmem) -> int32_t {
        if (p->dtype == SGL_DTYPE_F32) return 1;
        return std::min<int32_t>(Hkv, nmem * G <= 8 ? sgl::kDecHeadBlock : sgl::kDecHeadBlock / 2);
    };
    struct Unit {   // narrow work: one member block of a segment for a block of KV heads
        int32_t rep_row, b, e, kvh, mem_begin, n_mem, nh;
        bool tail;      // a request's own trailing positions: its last piece runs to seq_len at run time
    };
    // The plan's member list: the groups' members, then one entry per
    // request whose context does not end in a segment of its own (it ends
    // in a shared segment, or is empty); such a request gets an empty
    // trailing unit at its end, so that every request has a piece that
    // reads its positions past the planned length when the batch has grown
    // (decode steps reuse the plan; the kernels read seq_lens).
    std::vector<int32_t> mem(g->seg_members, g->seg_members + g->num_members);
    std::vector<int32_t> own_tail(B, -1);   // segment that is request r's own trailing segment
    for (int32_t s = 0; s < nseg; ++s) {
        const int32_t m0 = g->seg_member_ptr[s], m1 = g->seg_member_ptr[s + 1];
        if (m1 - m0 == 1 && g->seg_end[s] == seq_lens[g->seg_members[m0]]) own_tail[g->seg_members[m0]] = s;
    }
    std::vector<Unit> units;
    int64_t units_n = 0;     // position-heads
    int64_t max_wide = 0;
    auto add_units = [&](int32_t rep, int32_t b, int32_t e, int32_t m0, int32_t nmem, bool tail) {
        const int32_t HP = head_block(nmem);
        for (int32_t h = 0; h < Hkv; h += HP) {
            const int32_t nh = std::min(HP, Hkv - h);
            units.push_back({rep, b, e, h, m0, nmem, nh, tail});
            units_n += (int64_t)(e - b) * nh;
        }
    };
    for (int32_t s = 0; s < nseg; ++s) {
        const int32_t b = g->seg_begin[s], e = g->seg_end[s];
        const int32_t m0 = g->seg_member_ptr[s], nmem = g->seg_member_ptr[s + 1] - m0;
        if (nmem <= MBn)
            add_units(g->seg_row[s], b, e, m0, nmem, nmem == 1 && own_tail[g->seg_members[m0]] == s);
        else
            max_wide = std::max<int64_t>(max_wide, e - b);
    }
    for (int32_t r = 0; r < B; ++r) {
        if (own_tail[r] >= 0) continue;
        mem.push_back(r);
        add_units(r, seq_lens[r], seq_lens[r], (int32_t)mem.size() - 1, 1, true);
    }
    const int64_t n_ctas = sms;
    // Wide chunks run on tile CTAs whose streaming warps start only when
    // their tiles are done (so the two never compete for an SM's issue slots
    // and instruction cache); the other CTAs stream from the start.  Chunk
    // length and tile CTA count come from a cost model of this kernel on
    // GB300 (measured): a tile costs ~2 us plus ~2.5 us per 128-position
    // block; a streaming SM handles ~88 (d=128) position-heads per us after
    // ~4 us of start-up.  The chunk length with the earliest estimated finish
    // is taken (tile CTAs at most half the CTAs).
    auto wide_items_for = [&](int64_t Cw) {
        int64_t n = 0;
        for (int32_t s = 0; s < nseg; ++s) {
            const int32_t nmem = g->seg_member_ptr[s + 1] - g->seg_member_ptr[s];
            if (nmem > MBn)
                n += (g->seg_end[s] - g->seg_begin[s] + Cw - 1) / Cw * ((nmem + MBw - 1) / MBw) * Hkv;
        }
        return n;
    };
    const double rate = 88.0 * 128.0 / p->head_dim;   // streamed position-heads per us per SM
    int64_t Cw = 128, n_tile_ctas = 0;
    if (max_wide > 0) {
        double best = 1e300;
        const int64_t top = std::min<int64_t>((max_wide + 127) / 128 * 128, 128 * 256);
        for (int64_t c = 128; c <= top; c += 128) {
            const int64_t nw = wide_items_for(c);
            const int64_t T = std::max<int64_t>(1, std::min<int64_t>(nw, n_ctas / 2));
            const double per = (double)((nw + T - 1) / T);
            const double tile_us = per * (2.0 + 2.5 * (double)c / 128.0);
            // streaming CTAs work from ~5 us; a tile CTA streams only what is
            // left when its tiles are done, which the estimate ignores
            const double F = std::max(tile_us, 4.0 + (double)units_n /
                                                     ((double)std::max<int64_t>(1, n_ctas - T) * rate));
            if (F < best) {
                best = F;
                Cw = c;
                n_tile_ctas = T;
            }
        }
    }
    std::vector<sgl::DecItem> wide;
    for (int32_t s = 0; s < nseg; ++s) {
        const int32_t b = g->seg_begin[s], e = g->seg_end[s];
        const int32_t m0 = g->seg_member_ptr[s], nmem = g->seg_member_ptr[s + 1] - m0;
        if (nmem <= MBn) continue;
        const int32_t nblk = (nmem + MBw - 1) / MBw;
        for (int64_t cb = b; cb < e; cb += Cw) {
            const int32_t ce = (int32_t)std::min<int64_t>(e, cb + Cw);
            for (int32_t blk = 0; blk < nblk; ++blk) {
                const int32_t mb = blk * MBw, nm = std::min(MBw, nmem - mb);
                for (int32_t h = 0; h < Hkv; ++h)
                    wide.push_back({g->seg_row[s], (int32_t)cb, ce, h, m0 + mb, nm, 0, 1});
            }
        }
    }

    // Narrow units are cut into pieces of at most Pmax positions (about half
    // an even share of a stream, so that the run-time counter can balance
    // the tail; a cut makes one more partial to merge), no
    // piece shorter than one 16-position step unless its unit is, ordered
    // longest first.  Each streaming CTA starts on its own piece; the rest
    // (and all work of tile CTAs' streams, once their tiles are done) are
    // handed out at run time from a counter, so SMs that stream faster take
    // more.
    const int64_t n_cons = n_ctas - n_tile_ctas;
    // (in position-heads, so that a piece of a 4-head block is as long in
    // bytes as one of an 8-head block)
    const int64_t Pph = (int64_t)std::ceil((double)units_n / (double)std::max<int64_t>(1, 2 * n_cons));
    std::vector<std::pair<int32_t, sgl::DecItem>> cut;   // (planned length, piece)
    for (const Unit& u : units) {
        int64_t Pmax = (Pph + u.nh - 1) / u.nh;
        Pmax = std::min<int64_t>(2048, std::max<int64_t>(32, (Pmax + 15) / 16 * 16));
        for (int64_t pos = u.b; pos < u.e || (pos == u.b && u.tail);) {
            int64_t take = std::min<int64_t>(u.e - pos, Pmax);
            if (u.e - pos - take < 16) take = u.e - pos;   // no tail piece under one step
            const bool last = pos + take == u.e;
            cut.push_back({(int32_t)take,
                           {u.rep_row, (int32_t)pos, last && u.tail ? sgl::kDecToSeqEnd : (int32_t)(pos + take), u.kvh,
                            u.mem_begin, u.n_mem, 0, u.nh}});
            pos += take;
            if (take == 0) break;   // (an empty trailing unit: one piece)
        }
    }
    std::stable_sort(cut.begin(), cut.end(), [](const std::pair<int32_t, sgl::DecItem>& x,
                                                const std::pair<int32_t, sgl::DecItem>& y) {
        return x.first > y.first;
    });
    std::vector<sgl::DecItem> narrow;
    narrow.reserve(cut.size());
    for (const auto& c : cut) narrow.push_back(c.second);
    const int64_t n_init = std::min<int64_t>((int64_t)narrow.size(), n_cons);

    // wide items round-robin over the tile CTAs (the first n_tile_ctas)
    std::vector<std::vector<sgl::DecItem>> cta_items((size_t)n_ctas);
    for (size_t i = 0; i < wide.size(); ++i) cta_items[i % (size_t)std::max<int64_t>(1, n_tile_ctas)].push_back(wide[i]);

    // final item order: wide items by CTA, then the narrow pieces; partial
    // rows in item order
    std::vector<sgl::DecItem> items;
    std::vector<int32_t> wptr;
    wptr.push_back(0);
    for (auto& v : cta_items) {
        items.insert(items.end(), v.begin(), v.end());
        wptr.push_back((int32_t)items.size());
    }
    const int32_t n_wide = (int32_t)items.size();
    items.insert(items.end(), narrow.begin(), narrow.end());
    // merge lists of (request, KV head), entries in item order: counted,
    // then filled (one flat array)
    const size_t n_keys = (size_t)B * Hkv;
    std::vector<int32_t> eptr(n_keys + 1, 0);
    int64_t prow = 0;
    for (auto& it : items) {
        it.partial_base = (int32_t)prow;
        for (int32_t i = 0; i < it.n_mem; ++i)
            for (int32_t hh = 0; hh < it.nh; ++hh)
                ++eptr[(size_t)mem[it.mem_begin + i] * Hkv + it.kvh + hh + 1];
        prow += (int64_t)it.n_mem * it.nh * G;
        if (prow > INT32_MAX / 256) return SGL_ERR_UNSUPPORTED;
    }
    int32_t max_ent = 0;
    for (size_t k = 0; k < n_keys; ++k) {
        max_ent = std::max(max_ent, eptr[k + 1]);
        eptr[k + 1] += eptr[k];
    }
    const int64_t n_ent = eptr[n_keys];
    std::vector<int32_t> ents_flat((size_t)n_ent);
    {
        std::vector<int32_t> fill(eptr.begin(), eptr.end() - 1);
        for (const auto& it : items)
            for (int32_t i = 0; i < it.n_mem; ++i)
                for (int32_t hh = 0; hh < it.nh; ++hh)
                    ents_flat[fill[(size_t)mem[it.mem_begin + i] * Hkv + it.kvh + hh]++] =
                        it.partial_base + (i * it.nh + hh) * G;
    }

    sgl_plan* plan = new (std::nothrow) sgl_plan();
    if (!plan) return SGL_ERR_INVALID_ARG;
    plan->params = *p;
    plan->params.host_prefix_lens = nullptr;
    plan->params.host_extend_lens = nullptr;
    plan->G = G;
    plan->n_items = (int32_t)items.size();
    plan->n_wide = n_wide;
    plan->n_partial_rows = (int32_t)prow;
    plan->n_ctas = (int32_t)n_ctas;
    plan->n_narrow = (int32_t)narrow.size();
    plan->n_init = (int32_t)n_init;
    plan->n_tile_ctas = (int32_t)n_tile_ctas;
    plan->n_members = (int32_t)mem.size();
    plan->n_merge_entries = (int32_t)n_ent;
    plan->chunk_tokens = (int32_t)Cw;
    plan->max_pos = 0;
    for (int32_t s = 0; s < nseg; ++s) plan->max_pos = std::max(plan->max_pos, g->seg_end[s]);
    plan->max_entries_per_request = max_ent;

    using sgl::align_up;
    const size_t A = sgl::kWsAlign;
    plan->off_items = A;
    plan->off_members = align_up(plan->off_items + items.size() * sizeof(sgl::DecItem), A);
    plan->off_wptr = align_up(plan->off_members + mem.size() * 4, A);
    plan->off_sched = align_up(plan->off_wptr + wptr.size() * 4, A);
    plan->off_mptr = align_up(plan->off_sched + 2 * 4, A);
    plan->off_ment = align_up(plan->off_mptr + ((size_t)B * Hkv + 1) * 4, A);
    plan->tables_bytes = align_up(plan->off_ment + (size_t)n_ent * 4, A);
    plan->off_plse = plan->tables_bytes;
    plan->off_po = align_up(plan->off_plse + (size_t)prow * 4, A);
    plan->off_cnt = align_up(plan->off_po + (size_t)prow * p->head_dim * 4, A);
    plan->workspace_bytes = align_up(plan->off_cnt + (size_t)B * Hkv * 4, A);

    plan->blob = new (std::nothrow) unsigned char[plan->tables_bytes];
    if (!plan->blob) {
        delete plan;
        return SGL_ERR_INVALID_ARG;
    }
    std::memset(plan->blob, 0, plan->tables_bytes);
    sgl::WsHeader hdr{0u, sgl::kWsMagic, plan->n_items, plan->n_wide, plan->n_partial_rows, plan->n_ctas};
    std::memcpy(plan->blob, &hdr, sizeof(hdr));
    if (!items.empty()) std::memcpy(plan->blob + plan->off_items, items.data(), items.size() * sizeof(sgl::DecItem));
    if (!mem.empty()) std::memcpy(plan->blob + plan->off_members, mem.data(), mem.size() * 4);
    std::memcpy(plan->blob + plan->off_wptr, wptr.data(), wptr.size() * 4);
    // run-time piece counter: next piece to hand out, producers finished
    const uint32_t sched[2] = {(uint32_t)n_init, 0u};
    std::memcpy(plan->blob + plan->off_sched, sched, sizeof(sched));
    std::memcpy(plan->blob + plan->off_mptr, eptr.data(), eptr.size() * 4);
    if (n_ent) std::memcpy(plan->blob + plan->off_ment, ents_flat.data(), (size_t)n_ent * 4);
    *plan_out = plan;
    *workspace_bytes = plan->workspace_bytes;
    return SGL_OK;
}

void sgl_plan_destroy(sgl_plan* plan) {
    if (!plan) return;
    delete[] plan->blob;
    delete plan;
}

int sgl_plan_info(const sgl_plan* plan, sgl_plan_info_t* out) {
    if (!plan || !out) return SGL_ERR_INVALID_ARG;
    out->num_items = plan->n_items;
    out->num_wide_items = plan->n_wide;
    out->num_partial_rows = plan->n_partial_rows;
    out->num_merge_entries = plan->n_merge_entries;
    out->chunk_tokens = plan->chunk_tokens;
    out->upload_bytes = (int64_t)plan->tables_bytes;
    out->workspace_bytes = (int64_t)plan->workspace_bytes;
    return SGL_OK;
}

int sgl_extend_workspace_bytes(const sgl_attn_params* p, size_t* bytes) {
    int st = sgl::check_params(p);
    if (st) return st;
    if (!bytes) return SGL_ERR_INVALID_ARG;
    *bytes = sgl::kWsAlign;   // the error word
    return SGL_OK;
}

}  // extern "C"
