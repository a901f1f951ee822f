// Prefix-group scheduler for decode: turns the batch's prefix groups into
// GPU work items and the per-request merge lists.
//
// A segment (a run of positions shared by a set of member requests, read
// from one representative row) is the unit of sharing: its K/V are read
// once for all members and all query heads of a KV head -- "computed once,
// referenced many times" ("SGLang：从前端 DSL 到 SRT 服务运行时", section
// "用基数树实现前缀复用"; bhfrc.com/news/45689 §1.3).  The pages give no
// kernel schedule; this one is ours:
//   * a segment with at most 8 query rows (member x query head of a KV
//     head) is narrow: its chunks go to a one-warp-per-item kernel, chunk
//     length sized for ~24 warps of work per SM (>= 64 positions);
//   * a wider segment (a prefix shared by many requests) is split into member
//     blocks of up to 128 rows (one tensor-core tile), each chunk read once per
//     block by a CTA that stages it in shared memory (tcgen05 kernel), chunk
//     length a multiple of the 128-position KV block sized for ~1 CTA per SM;
//   * items are ordered chunk-major with the KV head innermost, so work that
//     runs together reads the heads of the same tokens (one token's K for
//     all heads is one contiguous row of the slot-major pool);
//   * each item writes its rows' normalised partial O and LSE (fp32); a
//     request's merge list names every partial row it must combine.

#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "common.h"

namespace {

int query_num_sms(int32_t requested) {
    if (requested > 0) return requested;
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
        return n;
    cudaGetLastError();
    return 152;
}

}  // namespace

namespace sgl {

int check_params(const sgl_attn_params* p) {
    if (!p) return SGL_ERR_INVALID_ARG;
    if (p->batch < 0 || p->num_qo_heads <= 0 || p->num_kv_heads <= 0 || p->num_slots < 0 || p->page_size < 1)
        return SGL_ERR_INVALID_ARG;
    if (p->dtype != SGL_DTYPE_F32 && p->dtype != SGL_DTYPE_BF16) return SGL_ERR_UNSUPPORTED;
    if (p->head_dim != 64 && p->head_dim != 128) return SGL_ERR_UNSUPPORTED;
    if (p->num_qo_heads % p->num_kv_heads) return SGL_ERR_UNSUPPORTED;
    int G = p->num_qo_heads / p->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return SGL_ERR_UNSUPPORTED;
    if (p->num_slots > INT32_MAX) return SGL_ERR_UNSUPPORTED;
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

    // Narrow segments (at most 8 query rows: member x query head of a KV
    // head) go to the one-warp-per-item kernel; wider ones to the CTA kernel
    // in member blocks of up to 64 rows.
    const int32_t MBn = std::max(1, 8 / G);
    const int32_t MBw = std::max(1, 128 / G);
    double units_n = 0, units_w = 0;
    for (int32_t s = 0; s < nseg; ++s) {
        const int32_t nmem = g->seg_member_ptr[s + 1] - g->seg_member_ptr[s];
        const double len = (double)(g->seg_end[s] - g->seg_begin[s]);
        if (nmem <= MBn)
            units_n += len * Hkv;
        else
            units_w += len * ((nmem + MBw - 1) / MBw) * Hkv;
    }
    const int sms = query_num_sms(p->num_sms);
    // narrow: ~24 warps of work per SM (16-position steps, chunks of >= 64)
    int64_t Cn = (int64_t)std::ceil(units_n / (24.0 * sms));
    Cn = std::max<int64_t>(64, (Cn + 15) / 16 * 16);
    // wide: ~1 CTA of work per SM (128-position KV blocks)
    int64_t Cw = (int64_t)std::ceil(units_w / (1.0 * sms));
    Cw = std::max<int64_t>(128, (Cw + 127) / 128 * 128);
    const int64_t C = Cn;

    std::vector<sgl::DecItem> wide, narrow;
    std::vector<std::vector<sgl::MergeEnt>> ents(B);
    int64_t prow = 0;
    for (int32_t s = 0; s < nseg; ++s) {
        const int32_t b = g->seg_begin[s], e = g->seg_end[s];
        const int32_t m0 = g->seg_member_ptr[s], nmem = g->seg_member_ptr[s + 1] - m0;
        const bool is_narrow = nmem <= MBn;
        const int32_t MB = is_narrow ? MBn : MBw;
        const int64_t CS = is_narrow ? Cn : Cw;
        const int32_t nblk = (nmem + MB - 1) / MB;
        for (int64_t cb = b; cb < e; cb += CS) {
            const int32_t ce = (int32_t)std::min<int64_t>(e, cb + CS);
            for (int32_t blk = 0; blk < nblk; ++blk) {
                const int32_t mb = blk * MB, nm = std::min(MB, nmem - mb);
                const int64_t base0 = prow;
                for (int32_t h = 0; h < Hkv; ++h) {
                    sgl::DecItem it;
                    it.rep_row = g->seg_row[s];
                    it.kv_begin = (int32_t)cb;
                    it.kv_end = ce;
                    it.kvh = h;
                    it.mem_begin = m0 + mb;
                    it.n_mem = nm;
                    it.partial_base = (int32_t)prow;
                    it.pad = 0;
                    (is_narrow ? narrow : wide).push_back(it);
                    prow += (int64_t)nm * G;
                }
                for (int32_t i = 0; i < nm; ++i) {
                    int32_t r = g->seg_members[m0 + mb + i];
                    ents[r].push_back({(int32_t)(base0 + (int64_t)i * G), nm * G});
                }
            }
        }
    }
    if (prow > INT32_MAX / 256) return SGL_ERR_UNSUPPORTED;
    std::vector<sgl::DecItem> items(wide);
    items.insert(items.end(), narrow.begin(), narrow.end());

    sgl_plan* plan = new (std::nothrow) sgl_plan();
    if (!plan) return SGL_ERR_INVALID_ARG;
    plan->params = *p;
    plan->params.host_prefix_lens = nullptr;
    plan->params.host_extend_lens = nullptr;
    plan->G = G;
    plan->n_items = (int32_t)items.size();
    plan->n_wide = (int32_t)wide.size();
    plan->n_partial_rows = (int32_t)prow;
    plan->n_members = g->num_members;
    int64_t n_ent = 0;
    int32_t max_ent = 0;
    for (auto& v : ents) {
        n_ent += (int64_t)v.size();
        max_ent = std::max<int32_t>(max_ent, (int32_t)v.size());
    }
    plan->n_merge_entries = (int32_t)n_ent;
    plan->chunk_tokens = (int32_t)C;
    plan->max_pos = 0;
    for (int32_t s = 0; s < nseg; ++s) plan->max_pos = std::max(plan->max_pos, g->seg_end[s]);
    plan->max_entries_per_request = max_ent;

    using sgl::align_up;
    const size_t A = sgl::kWsAlign;
    plan->off_items = A;
    plan->off_members = align_up(plan->off_items + items.size() * sizeof(sgl::DecItem), A);
    plan->off_mptr = align_up(plan->off_members + (size_t)g->num_members * 4, A);
    plan->off_ment = align_up(plan->off_mptr + (size_t)(B + 1) * 4, A);
    plan->tables_bytes = align_up(plan->off_ment + (size_t)n_ent * sizeof(sgl::MergeEnt), A);
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
    sgl::WsHeader hdr{0u, sgl::kWsMagic, plan->n_items, plan->n_partial_rows};
    std::memcpy(plan->blob, &hdr, sizeof(hdr));
    if (!items.empty()) std::memcpy(plan->blob + plan->off_items, items.data(), items.size() * sizeof(sgl::DecItem));
    if (g->num_members) std::memcpy(plan->blob + plan->off_members, g->seg_members, (size_t)g->num_members * 4);
    int32_t* mptr = reinterpret_cast<int32_t*>(plan->blob + plan->off_mptr);
    sgl::MergeEnt* ment = reinterpret_cast<sgl::MergeEnt*>(plan->blob + plan->off_ment);
    int64_t at = 0;
    for (int32_t r = 0; r < B; ++r) {
        mptr[r] = (int32_t)at;
        for (auto& e : ents[r]) ment[at++] = e;
    }
    mptr[B] = (int32_t)at;
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
