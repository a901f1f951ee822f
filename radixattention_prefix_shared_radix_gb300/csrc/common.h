// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include "sglattn.h"

namespace sgl {

// Record the cudaError_t behind an SGL_ERR_CUDA (thread-local).
void set_cuda_error(int err);

// SM count to plan for: `requested` if positive, else the current device's
// (152 when no device can be queried).
int query_num_sms(int32_t requested);

// Prefix groups of a batch of B requests checked against seq_lens (host):
// every request's segments tile [0, seq_len) exactly, members are sorted,
// every member holds the segment's positions, representatives are members.
// SGL_OK or SGL_ERR_INVALID_ARG.
int validate_groups(int32_t B, const int32_t* seq_lens, const sgl_prefix_groups* g);

// Decode work item: one KV chunk of one prefix-group segment for a block of
// `nh` consecutive KV heads and one block of the segment's members.  Laid out
// in the workspace.  Its query rows are ordered member, then KV head of the
// block, then query head of the group: row ((i * nh) + hh) * G + g is member
// i's query head (kvh + hh) * G + g, and partial row partial_base + row holds
// its result.
struct DecItem {
    int32_t rep_row;       // request row whose req_to_token slots are read
    int32_t kv_begin;      // first position of the chunk
    int32_t kv_end;        // one past the last position
    int32_t kvh;           // first KV head of the block
    int32_t mem_begin;     // first member in the plan's member array
    int32_t n_mem;         // members in this block
    int32_t partial_base;  // first partial row
    int32_t nh;            // KV heads in the block (1 for tensor-core tiles)
};
static_assert(sizeof(DecItem) == 32, "DecItem is 32 bytes");
// kv_end of a request's last piece (its own trailing positions): the piece
// runs to the request's seq_len at run time, so a plan stays valid while the
// batch's requests grow at their ends (decode steps).
constexpr int32_t kDecToSeqEnd = 0x7fffffff;

// Decode schedule constants (bf16 persistent kernel): a narrow piece covers
// up to kDecHeadBlock KV heads of its positions (one or two consumer warps
// each) for up to kDecPieceMembers member requests (the member slots of the
// kernel's lookup ring entry).
constexpr int kDecHeadBlock = 8;
constexpr int kDecPieceMembers = 8;

// Workspace header (first 256 bytes): error word + plan dimensions.
struct WsHeader {
    uint32_t error;        // bit 0: slot out of pool; bit 1: position beyond seq_len
    uint32_t magic;
    int32_t n_items;             // all work items: wide ones first, then narrow ones
    int32_t n_wide;              // items with more than 8 query rows (tcgen05 tiles)
    int32_t n_partial_rows;
    int32_t n_ctas;              // CTAs of the fused decode kernel
};
constexpr uint32_t kWsMagic = 0x53474c41u;  // "SGLA"
constexpr size_t kWsAlign = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace sgl

// Plan object (host); its tables are copied into the workspace head.
struct sgl_plan {
    int32_t kind;                // 0: GQA decode (sgl_decode_plan), 1: MLA decode (sgl_mla_decode_plan)
    sgl_attn_params params;      // host pointers cleared
    int32_t G;
    int32_t n_items;             // all work items: wide ones first, then narrow ones
    int32_t n_wide;              // items with more than 8 query rows (tcgen05 tiles)
    int32_t n_partial_rows;
    int32_t n_ctas;              // fused decode kernel: CTAs (wide items wptr[c]..wptr[c+1])
    int32_t n_narrow;            // narrow pieces (items n_wide .. n_items-1, longest first)
    int32_t n_init;              // pieces assigned at launch (streaming consumer w starts on piece w)
    int32_t n_tile_ctas;         // CTAs 0 .. n_tile_ctas-1 run the wide items, then stream
    int32_t n_members;
    int32_t n_merge_entries;
    int32_t max_entries_per_request;
    int32_t chunk_tokens;
    int32_t max_pos;             // largest segment end (req_to_token must have ld >= max_pos)
    // workspace offsets: items, members, wptr [n_ctas+1] (wide items of each
    // CTA), sched [2] (run-time piece counter and finished-producer count,
    // restored by the kernel), mptr [B*Hkv+1] and ment (first partial row of
    // each merge entry of (request, KV head)), then the fp32 partial LSEs and
    // rows and a spare counter area.
    size_t off_items, off_members, off_wptr, off_sched, off_mptr, off_ment, off_plse, off_po, off_cnt;
    size_t tables_bytes;         // bytes uploaded (header + tables)
    size_t workspace_bytes;      // total device workspace
    unsigned char* blob;         // host copy of [0, tables_bytes)
};

namespace sgl {
// The argument checks of sgl_decode_attn, all on the host, so that every
// refusal comes before any GPU work (shared with sgl_decode_step, which
// checks before its input copy).
inline int decode_arg_status(const sgl_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                             const int32_t* req_to_token, int64_t ld, const int32_t* seq_lens, const void* o,
                             const float* lse, const void* workspace, size_t ws_bytes) {
    auto aligned = [](const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
    if (!plan || plan->kind != 0) return SGL_ERR_INVALID_ARG;
    const int32_t B = plan->params.batch;
    if (B > 0 && (!q || !o || !lse || !seq_lens)) return SGL_ERR_INVALID_ARG;
    if (plan->n_items > 0 && (!k_pool || !v_pool || !req_to_token || ld < plan->max_pos)) return SGL_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, kWsAlign) || ws_bytes < plan->workspace_bytes) return SGL_ERR_WORKSPACE;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o, 16)) return SGL_ERR_INVALID_ARG;
    return SGL_OK;
}
}  // namespace sgl
