// Work items of the MLA grouped decode.
//
// MLA keeps ONE stored row per token (a 512-dim latent plus a 64-dim
// position part) that every query head reads (CS349D lecture-16 notes,
// SGLang case study, §4 "More engineering" and §5.1 "DP attention").  A
// prefix-group segment is therefore read once for all its member requests
// and all their query heads: the work unit is 64 query rows (member x head)
// of one segment chunk.  With Hq query heads a unit holds 64 / min(Hq, 64)
// members and min(Hq, 64) heads ("head group"; Hq = 128 has two groups of 64
// heads that read the same rows).  Two full units of one segment (e.g. two
// blocks of members sharing a prefix, or the two head groups of a request at
// Hq = 128) read the same rows: they are paired into a 128-row tcgen05 tile
// (mla_tile.cuh) run by two CTAs, one per half of the output columns; the
// other units run as mma.sync items.  Chunks are cut by a cost model of the
// kernel (measured on GB300: a 32-position block of a tile pair costs ~2.1 us
// per CTA after ~9 us of fixed cost; an item of at most 16 rows, e.g. a
// request's own suffix at Hq = 16, ~1.8 us per block after ~3.1 us; larger
// items ~0.94 us + 0.0394 us per query row per block after ~1.5 us); of the
// piece lengths tried, the planner keeps the
// one whose list schedule (items most costly first, each to the SM that
// frees first, as CTAs are dispatched) plus the traffic of its partial rows
// ends earliest.  Each item writes normalised partial rows that the
// log-sum-exp merge combines per (request, head group).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <new>
#include <queue>
#include <vector>

#include "common.h"

namespace {

constexpr int32_t kMlaRows = 64;    // query rows of one work item
constexpr int32_t kMlaBlock = 32;   // positions per block of the kernel

// estimated microseconds of one 32-position block for an item of `rows` query
// rows, and of an item's start (an item of at most 16 rows spreads each block
// over all 16 warps of the CTA: ~1.8 us per block after ~3.1 us, measured)
double block_cost(int32_t rows) { return rows <= 16 ? 1.785 : 0.94 + 0.0394 * rows; }
double item_start(int32_t rows) { return rows <= 16 ? 3.1 : 1.5; }
// tcgen05 tile pairs (two 64-row units, two CTAs): estimated microseconds of
// one 32-position block and of a tile's fixed cost (Q load and first
// gathers, ~6 us; epilogue, ~3 us), from GB300 timelines of the tiles
constexpr double kTileBlock = 2.1;
constexpr double kTileStart = 9.0;
// a partial row (512 fp32) is written by the kernel and read by the merge:
// 4 KB at about 6 TB/s
constexpr double kRowCost = 4096.0 / 6.0e6;

}  // namespace

extern "C" int sgl_mla_decode_plan(const sgl_mla_params* p, const int32_t* seq_lens, const sgl_prefix_groups* g,
                                   sgl_plan** plan_out, size_t* workspace_bytes) {
    if (!p || !g || !plan_out || !workspace_bytes) return SGL_ERR_INVALID_ARG;
    if (p->batch < 0 || p->num_slots < 0 || p->page_size < 1 || !(p->sm_scale >= 0.f) || std::isinf(p->sm_scale))
        return SGL_ERR_INVALID_ARG;
    if (p->latent_dim != 512 || p->rope_dim != 64) return SGL_ERR_UNSUPPORTED;
    const int32_t Hq = p->num_qo_heads;
    if (Hq != 16 && Hq != 32 && Hq != 64 && Hq != 128) return SGL_ERR_UNSUPPORTED;
    if (p->num_slots > INT32_MAX) return SGL_ERR_UNSUPPORTED;
    const int32_t B = p->batch;
    if (B > 0 && !seq_lens) return SGL_ERR_INVALID_ARG;
    int st = sgl::validate_groups(B, seq_lens, g);
    if (st) return st;

    const int32_t Gp = std::min<int32_t>(Hq, kMlaRows);   // heads per group
    const int32_t Hg = Hq / Gp;                           // head groups
    const int32_t MB = kMlaRows / Gp;                     // members per item
    const int32_t nseg = g->num_segments;
    const int sms = sgl::query_num_sms(p->num_sms);

    // Chunks: each (segment, member block, head group) unit is cut into
    // pieces of about T microseconds (whole blocks, at least two); T is
    // chosen among multiples of the mean work per SM by the end time of the
    // list schedule of the resulting items.
    struct Unit {
        int32_t s, mb, nm, hg;
        int64_t len;
        double per_block;   // per block of this unit (a pair: per block of each of its two CTAs)
        int32_t partner;    // the pair's second unit (this is the first), -1 single, -2 second of a pair
    };
    std::vector<Unit> units;
    double total = 0.0;
    for (int32_t s = 0; s < nseg; ++s) {
        const int32_t nmem = g->seg_member_ptr[s + 1] - g->seg_member_ptr[s];
        const int64_t len = g->seg_end[s] - g->seg_begin[s];
        const size_t first = units.size();
        for (int32_t mb = 0; mb < nmem; mb += MB)
            for (int32_t hg = 0; hg < Hg; ++hg) {
                const int32_t nm = std::min(MB, nmem - mb);
                units.push_back({s, mb, nm, hg, len, block_cost(nm * Gp), -1});
            }
        // pairs of full units of this segment, in order
        if (len >= 2 * kMlaBlock) {
            int32_t open = -1;
            for (size_t i = first; i < units.size(); ++i) {
                if (units[i].nm * Gp != kMlaRows) continue;
                if (open < 0) {
                    open = (int32_t)i;
                } else {
                    units[open].partner = (int32_t)i;
                    units[open].per_block = kTileBlock;
                    units[i].partner = -2;
                    open = -1;
                }
            }
        }
        for (size_t i = first; i < units.size(); ++i) {
            if (units[i].partner == -2) continue;
            const double ctas = units[i].partner >= 0 ? 2.0 : 1.0;
            total += ctas * units[i].per_block * (double)((len + kMlaBlock - 1) / kMlaBlock);
        }
    }
    auto pieces_of = [&](const Unit& u, double T) {   // blocks per piece, pieces
        const int64_t blocks = (u.len + kMlaBlock - 1) / kMlaBlock;
        const int64_t per = std::max<int64_t>(2, (int64_t)(T / u.per_block));
        const int64_t n = std::max<int64_t>(1, (blocks + per - 1) / per);
        return std::make_pair((blocks + n - 1) / n, n);
    };
    auto piece_costs = [&](double T, std::vector<double>& out) {
        out.clear();
        int64_t rows = 0;
        for (const Unit& u : units) {
            if (u.partner == -2) continue;
            const auto pc = pieces_of(u, T);
            const int64_t blocks = (u.len + kMlaBlock - 1) / kMlaBlock;
            for (int64_t k = 0; k < pc.second; ++k) {
                const int64_t nb = std::min(pc.first, blocks - k * pc.first);
                if (nb > 0) {
                    if (u.partner >= 0) {   // a tile piece: two CTAs
                        out.push_back(kTileStart + u.per_block * (double)nb);
                        out.push_back(kTileStart + u.per_block * (double)nb);
                        rows += 2 * kMlaRows;
                    } else {
                        out.push_back(item_start(u.nm * Gp) + u.per_block * (double)nb);
                        rows += (int64_t)u.nm * Gp;
                    }
                }
            }
        }
        std::sort(out.begin(), out.end(), std::greater<double>());
        return kRowCost * (double)rows;
    };
    auto makespan = [&](const std::vector<double>& c) {
        std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
        const size_t n_sm = std::min<size_t>((size_t)std::max(1, sms), std::max<size_t>(1, c.size()));
        for (size_t i = 0; i < n_sm; ++i) free_at.push(0.0);
        double end = 0.0;
        for (double x : c) {
            const double t = free_at.top() + x;
            free_at.pop();
            free_at.push(t);
            end = std::max(end, t);
        }
        return end;
    };
    const double mean = total / std::max(1, sms);
    double T = mean, best = INFINITY;
    size_t best_n = 0;
    std::vector<double> costs;
    for (int k = 0; k <= 64 && !units.empty(); ++k) {
        const double t = mean * (0.25 + 0.03 * k);
        const double merge = piece_costs(t, costs);
        const double m = makespan(costs) + merge;
        if (m < best * (1.0 - 1e-9) || (m <= best * (1.0 + 1e-9) && costs.size() < best_n)) {
            best = m;
            best_n = costs.size();
            T = t;
        }
    }
    struct Piece {
        sgl::DecItem item, second;   // second: the pair's other unit (tile pieces)
        double cost;
    };
    std::vector<Piece> pieces, tiles;
    int64_t C = 0;   // longest piece (reported as the chunk length)
    for (const Unit& u : units) {
        if (u.partner == -2) continue;
        const auto pc = pieces_of(u, T);
        const int64_t plen = pc.first * kMlaBlock;
        C = std::max(C, plen);
        const int32_t b = g->seg_begin[u.s], e = g->seg_end[u.s];
        for (int64_t cb = b; cb < e; cb += plen) {
            const int32_t ce = (int32_t)std::min<int64_t>(e, cb + plen);
            const int64_t nb = (ce - cb + kMlaBlock - 1) / kMlaBlock;
            const sgl::DecItem it{g->seg_row[u.s], (int32_t)cb, ce, u.hg, g->seg_member_ptr[u.s] + u.mb, u.nm, 0, 1};
            if (u.partner >= 0) {
                const Unit& v = units[(size_t)u.partner];
                const sgl::DecItem it2{g->seg_row[v.s], (int32_t)cb, ce, v.hg, g->seg_member_ptr[v.s] + v.mb, v.nm, 0, 1};
                tiles.push_back({it, it2, kTileStart + u.per_block * (double)nb});
            } else {
                pieces.push_back({it, it, item_start(u.nm * Gp) + u.per_block * (double)nb});
            }
        }
    }
    auto by_cost = [](const Piece& x, const Piece& y) { return x.cost > y.cost; };
    std::stable_sort(tiles.begin(), tiles.end(), by_cost);
    std::stable_sort(pieces.begin(), pieces.end(), by_cost);
    // items: the tile pieces' two units each (CTAs 2 t and 2 t + 1 both run
    // tile t, one output half each), then the mma.sync pieces
    std::vector<sgl::DecItem> items;
    items.reserve(2 * tiles.size() + pieces.size());
    for (const Piece& pc : tiles) {
        items.push_back(pc.item);
        items.push_back(pc.second);
    }
    for (const Piece& pc : pieces) items.push_back(pc.item);
    // partial rows in item order: member i of the item, head j of its group
    // at partial_base + i * Gp + j; merge lists per (request, head group)
    std::vector<std::vector<int32_t>> ents((size_t)B * Hg);
    int64_t prow = 0;
    for (auto& it : items) {
        it.partial_base = (int32_t)prow;
        for (int32_t i = 0; i < it.n_mem; ++i) {
            const int32_t r = g->seg_members[it.mem_begin + i];
            ents[(size_t)r * Hg + it.kvh].push_back((int32_t)(prow + (int64_t)i * Gp));
        }
        prow += (int64_t)it.n_mem * Gp;
        if (prow > INT32_MAX / 1024) return SGL_ERR_UNSUPPORTED;
    }
    if (items.size() > (size_t)INT32_MAX) return SGL_ERR_UNSUPPORTED;

    sgl_plan* plan = new (std::nothrow) sgl_plan();
    if (!plan) return SGL_ERR_INVALID_ARG;
    plan->kind = 1;
    sgl_attn_params& ap = plan->params;
    ap.dtype = SGL_DTYPE_BF16;
    ap.batch = B;
    ap.num_qo_heads = Hq;
    ap.num_kv_heads = Hg;
    ap.head_dim = p->latent_dim;
    ap.page_size = p->page_size;
    ap.num_slots = p->num_slots;
    ap.sm_scale = p->sm_scale > 0.f ? p->sm_scale : (float)(1.0 / std::sqrt((double)(p->latent_dim + p->rope_dim)));
    ap.num_sms = p->num_sms;
    plan->G = Gp;
    plan->n_items = (int32_t)items.size();
    plan->n_wide = (int32_t)(2 * tiles.size());   // tile CTAs (items 0 .. n_wide - 1, two per tile)
    plan->n_partial_rows = (int32_t)prow;
    plan->n_ctas = plan->n_items;
    plan->n_members = g->num_members;
    int64_t n_ent = 0;
    int32_t max_ent = 0;
    for (auto& v : ents) {
        n_ent += (int64_t)v.size();
        max_ent = std::max<int32_t>(max_ent, (int32_t)v.size());
    }
    plan->n_merge_entries = (int32_t)n_ent;
    plan->max_entries_per_request = max_ent;
    plan->chunk_tokens = (int32_t)C;
    plan->max_pos = 0;
    for (int32_t s = 0; s < nseg; ++s) plan->max_pos = std::max(plan->max_pos, g->seg_end[s]);

    using sgl::align_up;
    const size_t A = sgl::kWsAlign;
    plan->off_items = A;
    plan->off_members = align_up(plan->off_items + items.size() * sizeof(sgl::DecItem), A);
    plan->off_wptr = align_up(plan->off_members + (size_t)g->num_members * 4, A);
    plan->off_sched = plan->off_wptr;
    plan->off_mptr = align_up(plan->off_sched + 2 * 4, A);
    plan->off_ment = align_up(plan->off_mptr + ((size_t)B * Hg + 1) * 4, A);
    plan->tables_bytes = align_up(plan->off_ment + (size_t)n_ent * 4, A);
    plan->off_plse = plan->tables_bytes;
    plan->off_po = align_up(plan->off_plse + (size_t)prow * 4, A);
    plan->off_cnt = align_up(plan->off_po + (size_t)prow * p->latent_dim * 4, A);
    plan->workspace_bytes = align_up(plan->off_cnt + (size_t)B * Hg * 4, A);

    plan->blob = new (std::nothrow) unsigned char[plan->tables_bytes];
    if (!plan->blob) {
        delete plan;
        return SGL_ERR_INVALID_ARG;
    }
    std::memset(plan->blob, 0, plan->tables_bytes);
    sgl::WsHeader hdr{0u, sgl::kWsMagic, plan->n_items, plan->n_wide, plan->n_partial_rows, plan->n_ctas};
    std::memcpy(plan->blob, &hdr, sizeof(hdr));
    if (!items.empty()) std::memcpy(plan->blob + plan->off_items, items.data(), items.size() * sizeof(sgl::DecItem));
    if (g->num_members) std::memcpy(plan->blob + plan->off_members, g->seg_members, (size_t)g->num_members * 4);
    int32_t* mptr = reinterpret_cast<int32_t*>(plan->blob + plan->off_mptr);
    int32_t* ment = reinterpret_cast<int32_t*>(plan->blob + plan->off_ment);
    int64_t at = 0;
    for (size_t i = 0; i < ents.size(); ++i) {
        mptr[i] = (int32_t)at;
        for (int32_t e : ents[i]) ment[at++] = e;
    }
    mptr[ents.size()] = (int32_t)at;
    *plan_out = plan;
    *workspace_bytes = plan->workspace_bytes;
    return SGL_OK;
}
