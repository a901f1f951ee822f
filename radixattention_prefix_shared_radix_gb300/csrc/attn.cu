// GPU entry points of the C ABI, and the fp32 kernels.
//
// Decode ("SGLang 深度拆解" (chenxutan.com/d/5669.html) §3.2 PagedDecode and
// §4.1: one query token against the whole history, memory-bound) is split
// along the KV sequence into the planner's work items: a chunk of a prefix-
// group segment is read once for all its member requests and all query heads
// of a KV head ("computed once, referenced many times", "SGLang：从前端 DSL 到
// SRT 服务运行时", section "用基数树实现前缀复用").  Each item writes normalised
// partial rows (O, LSE) that a log-sum-exp merge combines per (request, head).
//   * bf16: the persistent decode kernel (decode_fused.cu): tcgen05 tiles
//     for shared segments beside producer/consumer streaming warps for the
//     rest; then the merge launch, one warp per (request, KV head).
//   * fp32 (exact CUDA-core arithmetic): one CTA per work item, then a merge
//     launch, one warp per (request, KV head).
//
// Extend ("SGLang 深度拆解" §3.2 PagedPrefill; "SGLang 深度解读" section
// "5. Attention 层": the new tokens' K/V are in the pool before attention):
// bf16 on the tcgen05 tile kernel (tc_attn.cu), fp32 one warp per
// (new token, query head).
//
// Softmax runs in base 2 on scores pre-multiplied by sm_scale * log2(e);
// LSE is returned in natural log.  Slots outside the pool are skipped and
// flagged in the workspace error word; nothing traps.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.h"
#include "device_common.cuh"
#include "merge.cuh"

namespace sgl {
template <int D, bool F8>
int launch_decode_fused(const sgl_plan* plan, const void* q, const void* kp, const void* vp, const int32_t* r2t,
                        int64_t ld, const int32_t* seq_lens, void* o, float* lse, unsigned char* ws, float scale_log2,
                        cudaStream_t s);
template <int D, bool F8>
int launch_extend_tc(const void* q, const void* kp, const void* vp, const void* kn, const void* vn, void* kw, void* vw,
                     const int32_t* r2t, int64_t ld, const int32_t* pre, const int32_t* ext, int B, int64_t n_rows,
                     int64_t tiles, void* o, float* lse, uint32_t* err, int Hq, int Hkv, int64_t num_slots,
                     float scale_log2, float k_scale, float v_scale, cudaStream_t s);
}  // namespace sgl

namespace {

using namespace sgldev;

// ---------------------------------------------------------------------------
// KV write into FP8 pools: each new bf16 K/V element goes to its slot as the
// E4M3 code of value / scale (IEEE fp32 division), rounded to nearest even
// and saturated to the largest finite E4M3 value (cvt.rn.satfinite), one
// thread per 8 elements.  Out-of-pool slots are skipped and set bit 0 of the
// error word.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
    return h;
}
__global__ void kv_scatter_e4m3(const uint4* __restrict__ kn, const uint4* __restrict__ vn, uint2* __restrict__ kw,
                                uint2* __restrict__ vw, const int32_t* __restrict__ r2t, int64_t ld,
                                const int32_t* __restrict__ pre, const int32_t* __restrict__ ext, int B, int64_t n_rows,
                                int Hkv, int chunks, int64_t num_slots, uint32_t* err, float k_scale, float v_scale) {
    const int64_t per_row = (int64_t)Hkv * chunks;   // 8-element groups per token row
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_rows * per_row * 2;
         i += (int64_t)gridDim.x * blockDim.x) {
        const bool v = i >= n_rows * per_row;
        const int64_t k = v ? i - n_rows * per_row : i;
        const int64_t row = k / per_row, within = k - row * per_row;
        int r = 0;
        int64_t acc = 0;
        for (; r < B; ++r) {
            const int e = __ldg(ext + r);
            if (row < acc + e) break;
            acc += e;
        }
        if (r >= B) continue;
        const int32_t sl = __ldg(r2t + (int64_t)r * ld + __ldg(pre + r) + (row - acc));
        if (sl < 0 || sl >= num_slots) {
            if (within == 0) atomicOr(err, 1u);
            continue;
        }
        const uint4 x = __ldg((v ? vn : kn) + row * per_row + within);
        const float sc = v ? v_scale : k_scale;
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            c[j] = e4m3x2_of(__fdiv_rn(__uint_as_float(w[j] << 16), sc),
                             __fdiv_rn(__uint_as_float(w[j] & 0xffff0000u), sc));
        (v ? vw : kw)[(int64_t)sl * per_row + within] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    }
}

// ---------------------------------------------------------------------------
// Decode partial kernel (fp32, CUDA cores, no tensor cores): one warp per
// query row of the item, 32 positions at a time with one position per lane:
// each lane takes its position's whole dot product (exact fp32 FFMA, the
// query row broadcast from shared memory), the warp combines the 32 scores
// with shuffles, and for O the lanes split head_dim and run over the 32
// positions, whose V rows are all independent loads.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128)
    decode_partial_f32(const float* __restrict__ q, const float* __restrict__ kp, const float* __restrict__ vp,
                       const int32_t* __restrict__ r2t, int64_t ld, const int32_t* __restrict__ seq_lens,
                       const sgl::DecItem* __restrict__ items, const int32_t* __restrict__ members,
                       float* __restrict__ po, float* __restrict__ plse, uint32_t* __restrict__ err, int Hq, int Hkv,
                       int G, int64_t num_slots, float scale_log2) {
    constexpr int E = D / 32;   // O columns per lane
    __shared__ __align__(16) float qs[4][D];
    const sgl::DecItem it = items[blockIdx.x];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rows = it.n_mem * it.nh * G;
    int kv_end = it.kv_end;
    const int rep_len = __ldg(seq_lens + it.rep_row);
    if (kv_end == sgl::kDecToSeqEnd) {   // a request's trailing piece: to its length now (within its row)
        kv_end = rep_len;
        if (kv_end > ld || kv_end < it.kv_begin) {
            if (threadIdx.x == 0) atomicOr(err, 2u);
            kv_end = kv_end > ld ? (int)ld : it.kv_begin;
        }
    } else if (kv_end > rep_len) {
        if (threadIdx.x == 0) atomicOr(err, 2u);
        kv_end = rep_len;
    }
    for (int r = warp; r < rows; r += 4) {
        // row r: member r / (nh G), KV head kvh + (r / G) % nh, query head r % G of its group
        const int mem = __ldg(members + it.mem_begin + r / (it.nh * G));
        const int kvh = it.kvh + (r / G) % it.nh;
        const float* qr = q + ((int64_t)mem * Hq + kvh * G + r % G) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) qs[warp][lane + 32 * e] = qr[lane + 32 * e];
        __syncwarp();
        const float4* q4 = reinterpret_cast<const float4*>(qs[warp]);
        float o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = 0.f;
        float m = -INFINITY, l = 0.f;
        for (int p0 = it.kv_begin; p0 < kv_end; p0 += 32) {
            const int p = p0 + lane;
            const int64_t slot = p < kv_end ? load_slot(r2t, ld, it.rep_row, p, num_slots, err) : -1;
            float s = -INFINITY;
            if (slot >= 0) {
                const float4* kr = reinterpret_cast<const float4*>(kp + (slot * Hkv + kvh) * D);
                float dot = 0.f;
#pragma unroll
                for (int c = 0; c < D / 4; ++c) {
                    const float4 k4 = __ldg(kr + c), q4c = q4[c];
                    dot = fmaf(q4c.x, k4.x, dot);
                    dot = fmaf(q4c.y, k4.y, dot);
                    dot = fmaf(q4c.z, k4.z, dot);
                    dot = fmaf(q4c.w, k4.w, dot);
                }
                s = dot * scale_log2;
            }
            float cmax = s;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, off));
            const float mn = fmaxf(m, cmax);
            if (mn == -INFINITY) continue;   // nothing in this chunk (nor before)
            const float a = exp2f(m - mn);   // 0 while nothing was accumulated
            const float pj = exp2f(s - mn);  // 0 for masked positions
            float psum = pj;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l = l * a + psum;
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] *= a;
#pragma unroll 8
            for (int j = 0; j < 32; ++j) {
                const float pb = __shfl_sync(0xffffffffu, pj, j);
                const int64_t sj = __shfl_sync(0xffffffffu, slot, j);
                if (sj >= 0) {
                    const float* vr = vp + (sj * Hkv + kvh) * D;
#pragma unroll
                    for (int e = 0; e < E; ++e) o[e] = fmaf(pb, __ldg(vr + lane + 32 * e), o[e]);
                }
            }
            m = mn;
        }
        const int64_t prow = (int64_t)it.partial_base + r;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) po[prow * D + lane + 32 * e] = o[e] * inv;
        if (lane == 0) plse[prow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        __syncwarp();   // qs[warp] is rewritten for the next row
    }
}

// ---------------------------------------------------------------------------
// Extend (fp32, CUDA cores): one warp per (new token, query head).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128)
    extend_f32(const float* __restrict__ qn, const float* __restrict__ kp, const float* __restrict__ vp,
               const int32_t* __restrict__ r2t, int64_t ld, const int32_t* __restrict__ prefix_lens,
               const int32_t* __restrict__ extend_lens, float* __restrict__ o, float* __restrict__ lse,
               uint32_t* __restrict__ err, int B, int Hq, int Hkv, int G, int64_t num_slots, int64_t n_rows,
               float scale_log2) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);   // (new row, head)
    const int h = (int)(w % Hq);
    const int64_t nrow = w / Hq;
    if (nrow >= n_rows) return;
    int req = -1, acc = 0;
    for (int r = 0; r < B; ++r) {
        const int e = __ldg(extend_lens + r);
        if (nrow < acc + e) {
            req = r;
            break;
        }
        acc += e;
    }
    if (req < 0) return;
    const int i = (int)(nrow - acc);
    const int pre = __ldg(prefix_lens + req);
    if (pre < 0 || (int64_t)pre + __ldg(extend_lens + req) > ld) {
        if (lane == 0) atomicOr(err, 2u);
        return;
    }
    const int lim = pre + i;
    const int kvh = h / G;
    const float* qr = qn + (nrow * Hq + h) * D + lane * E;
    float qv[E], ov[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qv[e] = qr[e];
        ov[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int pos = 0; pos <= lim; ++pos) {
        const int64_t slot = load_slot(r2t, ld, req, pos, num_slots, err);
        if (slot < 0) continue;
        const float* kr = kp + (slot * Hkv + kvh) * D + lane * E;
        const float* vr = vp + (slot * Hkv + kvh) * D + lane * E;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot = fmaf(qv[e], kr[e], dot);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float s = dot * scale_log2;
        const float mn = fmaxf(m, s);
        const float a = exp2f(m - mn), p = exp2f(s - mn);
        l = l * a + p;
#pragma unroll
        for (int e = 0; e < E; ++e) ov[e] = fmaf(p, vr[e], ov[e] * a);
        m = mn;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[(nrow * Hq + h) * D + lane * E + e] = ov[e] * inv;
    if (lane == 0) lse[nrow * Hq + h] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// KV write (fp32 path): new token i of request r -> pool slot
// req_to_token[r, prefix_len + i], for K and V, `rb` bytes per (token, head)
// row, one thread per 16-byte chunk.  Out-of-pool slots are skipped and set
// bit 0 of the error word.
__global__ void kv_scatter(const uint4* __restrict__ kn, const uint4* __restrict__ vn, uint4* __restrict__ kw,
                           uint4* __restrict__ vw, const int32_t* __restrict__ r2t, int64_t ld,
                           const int32_t* __restrict__ pre, const int32_t* __restrict__ ext, int B, int64_t n_rows,
                           int Hkv, int chunks, int64_t num_slots, uint32_t* err) {
    const int64_t per_row = (int64_t)Hkv * chunks;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_rows * per_row * 2;
         i += (int64_t)gridDim.x * blockDim.x) {
        const bool v = i >= n_rows * per_row;
        const int64_t k = v ? i - n_rows * per_row : i;
        const int64_t row = k / per_row, within = k - row * per_row;
        // request of this new-token row
        int r = 0;
        int64_t acc = 0;
        for (; r < B; ++r) {
            const int e = __ldg(ext + r);
            if (row < acc + e) break;
            acc += e;
        }
        if (r >= B) continue;
        const int32_t sl = __ldg(r2t + (int64_t)r * ld + __ldg(pre + r) + (row - acc));
        if (sl < 0 || sl >= num_slots) {
            if (within == 0) atomicOr(err, 1u);
            continue;
        }
        (v ? vw : kw)[(int64_t)sl * per_row + within] = (v ? vn : kn)[row * per_row + within];
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
thread_local int t_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SGL_OK;
    t_last_cuda_error = static_cast<int>(e);
    return SGL_ERR_CUDA;
}

float scale_log2_of(const sgl_attn_params* p) {
    const float sc = p->sm_scale > 0.f ? p->sm_scale : 1.0f / std::sqrt(static_cast<float>(p->head_dim));
    return sc * kLog2e;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <int D>
int launch_decode(const sgl_plan* plan, const void* q, const void* kp, const void* vp, const int32_t* r2t,
                  int64_t ld, const int32_t* seq_lens, void* o, float* lse, unsigned char* ws, cudaStream_t s) {
    const sgl_attn_params& p = plan->params;
    const float sl2 = scale_log2_of(&p);
    if (p.batch == 0) return SGL_OK;
    if (p.dtype == SGL_DTYPE_BF16 || p.dtype == SGL_DTYPE_BF16_FP8KV) {
        const int e = p.dtype == SGL_DTYPE_BF16
                          ? sgl::launch_decode_fused<D, false>(plan, q, kp, vp, r2t, ld, seq_lens, o, lse, ws, sl2, s)
                          : sgl::launch_decode_fused<D, true>(plan, q, kp, vp, r2t, ld, seq_lens, o, lse, ws, sl2, s);
        if (e) return cuda_status(static_cast<cudaError_t>(e));
        return SGL_OK;
    }
    const auto* items = reinterpret_cast<const sgl::DecItem*>(ws + plan->off_items);
    const auto* members = reinterpret_cast<const int32_t*>(ws + plan->off_members);
    float* plse = reinterpret_cast<float*>(ws + plan->off_plse);
    float* po = reinterpret_cast<float*>(ws + plan->off_po);
    uint32_t* err = reinterpret_cast<uint32_t*>(ws);
    const int Hq = p.num_qo_heads, Hkv = p.num_kv_heads, G = plan->G;
    if (plan->n_items > 0)
        decode_partial_f32<D><<<plan->n_items, 128, 0, s>>>(
            static_cast<const float*>(q), static_cast<const float*>(kp), static_cast<const float*>(vp), r2t, ld,
            seq_lens, items, members, po, plse, err, Hq, Hkv, G, p.num_slots, sl2);
    sgl::MergeArgs m{po, plse, reinterpret_cast<const int32_t*>(ws + plan->off_mptr),
                     reinterpret_cast<const int32_t*>(ws + plan->off_ment), o, lse, Hq, Hkv, G};
    const int n_pairs = p.batch * Hkv;
    sgl::decode_merge_kernel<float, D><<<sgl::merge_blocks<D>(n_pairs, G), 128, 0, s>>>(m, n_pairs);
    return cuda_status(cudaGetLastError());
}

template <int D>
int launch_extend(const sgl_attn_params* p, const void* q, const void* kp, const void* vp, const void* kn,
                  const void* vn, void* kw, void* vw, const int32_t* r2t, int64_t ld, const int32_t* pre,
                  const int32_t* ext, void* o, float* lse, uint32_t* err, cudaStream_t s) {
    const int Hq = p->num_qo_heads, Hkv = p->num_kv_heads, G = Hq / Hkv, B = p->batch;
    const float sl2 = scale_log2_of(p);
    int64_t total_rows = 0, tiles = 0;
    const int tq = 128 / G;
    for (int r = 0; r < B; ++r) {
        total_rows += p->host_extend_lens[r];
        tiles += ((p->host_extend_lens[r] + tq - 1) / tq + 1) / 2;   // CTAs: pairs of query tiles
    }
    if (total_rows == 0) return SGL_OK;
    if (p->dtype == SGL_DTYPE_BF16 || p->dtype == SGL_DTYPE_BF16_FP8KV) {
        if (tiles > INT32_MAX) return SGL_ERR_UNSUPPORTED;
        if (p->dtype == SGL_DTYPE_BF16_FP8KV && kn) {
            // FP8 pools: the new rows are quantised into the pool first, and
            // the extend then reads every position from the pool (so the new
            // block is attended at its stored, quantised values)
            kv_scatter_e4m3<<<1024, 256, 0, s>>>(static_cast<const uint4*>(kn), static_cast<const uint4*>(vn),
                                                 static_cast<uint2*>(kw), static_cast<uint2*>(vw), r2t, ld, pre, ext,
                                                 B, total_rows, Hkv, D / 8, p->num_slots, err, p->k_scale,
                                                 p->v_scale);
            kn = vn = nullptr;
            kw = vw = nullptr;
        }
        const int e = p->dtype == SGL_DTYPE_BF16_FP8KV
                          ? sgl::launch_extend_tc<D, true>(q, kp, vp, kn, vn, kw, vw, r2t, ld, pre, ext, B, total_rows,
                                                           tiles, o, lse, err, Hq, Hkv, p->num_slots, sl2, p->k_scale,
                                                           p->v_scale, s)
                          : sgl::launch_extend_tc<D, false>(q, kp, vp, kn, vn, kw, vw, r2t, ld, pre, ext, B, total_rows,
                                                            tiles, o, lse, err, Hq, Hkv, p->num_slots, sl2, 1.f, 1.f, s);
        if (e) return cuda_status(static_cast<cudaError_t>(e));
    } else {
        if (kn) {
            // the new K/V into the pool first (the exact path reads the pool)
            const int chunks = D * 4 / 16;
            kv_scatter<<<1024, 256, 0, s>>>(static_cast<const uint4*>(kn), static_cast<const uint4*>(vn),
                                            static_cast<uint4*>(kw), static_cast<uint4*>(vw), r2t, ld, pre, ext, B,
                                            total_rows, Hkv, chunks, p->num_slots, err);
        }
        const int64_t warps = total_rows * Hq;
        if ((warps + 3) / 4 > INT32_MAX) return SGL_ERR_UNSUPPORTED;
        extend_f32<D><<<static_cast<unsigned>((warps + 3) / 4), 128, 0, s>>>(
            static_cast<const float*>(q), static_cast<const float*>(kp), static_cast<const float*>(vp), r2t, ld, pre,
            ext, static_cast<float*>(o), lse, err, B, Hq, Hkv, G, p->num_slots, total_rows, sl2);
    }
    return cuda_status(cudaGetLastError());
}

}  // namespace

namespace sgl {
int check_params(const sgl_attn_params* p);
void set_cuda_error(int err) { t_last_cuda_error = err; }
}  // namespace sgl

extern "C" {

int sgl_last_cuda_error(void) { return t_last_cuda_error; }

int sgl_plan_upload(const sgl_plan* plan, void* workspace, size_t ws_bytes, sgl_stream_t stream) {
    if (!plan || !workspace) return SGL_ERR_INVALID_ARG;
    if (!aligned(workspace, sgl::kWsAlign) || ws_bytes < plan->workspace_bytes) return SGL_ERR_WORKSPACE;
    auto s = reinterpret_cast<cudaStream_t>(stream);
    int st = cuda_status(cudaMemcpyAsync(workspace, plan->blob, plan->tables_bytes, cudaMemcpyHostToDevice, s));
    if (st) return st;
    // merge counters start at zero (each merge resets its counter afterwards)
    return cuda_status(cudaMemsetAsync(static_cast<unsigned char*>(workspace) + plan->off_cnt, 0,
                                       plan->workspace_bytes - plan->off_cnt, s));
}

int sgl_decode_attn(const void* q, const void* k_pool, const void* v_pool, const int32_t* req_to_token, int64_t ld,
                    const int32_t* seq_lens, const sgl_plan* plan, void* o, float* lse, void* workspace,
                    size_t ws_bytes, sgl_stream_t stream) {
    if (const int st = sgl::decode_arg_status(plan, q, k_pool, v_pool, req_to_token, ld, seq_lens, o, lse, workspace,
                                              ws_bytes))
        return st;
    auto* ws = static_cast<unsigned char*>(workspace);
    auto s = reinterpret_cast<cudaStream_t>(stream);
    if (plan->params.head_dim == 128) return launch_decode<128>(plan, q, k_pool, v_pool, req_to_token, ld, seq_lens, o, lse, ws, s);
    return launch_decode<64>(plan, q, k_pool, v_pool, req_to_token, ld, seq_lens, o, lse, ws, s);
}

static int extend_impl(const void* q_new, const void* k_new, const void* v_new, const void* k_pool,
                       const void* v_pool, void* k_pool_w, void* v_pool_w, const int32_t* req_to_token, int64_t ld,
                       const int32_t* prefix_lens, const int32_t* extend_lens, const sgl_attn_params* params, void* o,
                       float* lse, void* workspace, size_t ws_bytes, sgl_stream_t stream) {
    int st = sgl::check_params(params);
    if (st) return st;
    const int32_t B = params->batch;
    if (B > 0 && (!params->host_extend_lens || !params->host_prefix_lens || !prefix_lens || !extend_lens))
        return SGL_ERR_INVALID_ARG;
    int64_t rows = 0;
    for (int32_t r = 0; r < B; ++r) {
        if (params->host_extend_lens[r] < 0 || params->host_prefix_lens[r] < 0) return SGL_ERR_INVALID_ARG;
        if ((int64_t)params->host_prefix_lens[r] + params->host_extend_lens[r] > ld) return SGL_ERR_INVALID_ARG;
        rows += params->host_extend_lens[r];
    }
    if (rows > 0 && (!q_new || !k_pool || !v_pool || !req_to_token || !o || !lse)) return SGL_ERR_INVALID_ARG;
    if (rows > 0 && k_new && (!v_new || !aligned(k_new, 16) || !aligned(v_new, 16))) return SGL_ERR_INVALID_ARG;
    if (rows * params->num_kv_heads > INT32_MAX) return SGL_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, sgl::kWsAlign) || ws_bytes < sgl::kWsAlign) return SGL_ERR_WORKSPACE;
    if (!aligned(q_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o, 16))
        return SGL_ERR_INVALID_ARG;
    auto s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t* err = static_cast<uint32_t*>(workspace);
    if (params->head_dim == 128)
        return launch_extend<128>(params, q_new, k_pool, v_pool, k_new, v_new, k_pool_w, v_pool_w, req_to_token, ld,
                                  prefix_lens, extend_lens, o, lse, err, s);
    return launch_extend<64>(params, q_new, k_pool, v_pool, k_new, v_new, k_pool_w, v_pool_w, req_to_token, ld,
                             prefix_lens, extend_lens, o, lse, err, s);
}

int sgl_extend_attn(const void* q_new, const void* k_pool, const void* v_pool, const int32_t* req_to_token,
                    int64_t ld, const int32_t* prefix_lens, const int32_t* extend_lens, const sgl_attn_params* params,
                    void* o, float* lse, void* workspace, size_t ws_bytes, sgl_stream_t stream) {
    return extend_impl(q_new, nullptr, nullptr, k_pool, v_pool, nullptr, nullptr, req_to_token, ld, prefix_lens,
                       extend_lens, params, o, lse, workspace, ws_bytes, stream);
}

int sgl_extend_attn_kvwrite(const void* q_new, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                            const int32_t* req_to_token, int64_t ld, const int32_t* prefix_lens,
                            const int32_t* extend_lens, const sgl_attn_params* params, void* o, float* lse,
                            void* workspace, size_t ws_bytes, sgl_stream_t stream) {
    if (params && params->batch > 0 && (!k_new || !v_new)) return SGL_ERR_INVALID_ARG;
    return extend_impl(q_new, k_new, v_new, k_pool, v_pool, k_pool, v_pool, req_to_token, ld, prefix_lens, extend_lens,
                       params, o, lse, workspace, ws_bytes, stream);
}

int sgl_check(void* workspace, sgl_stream_t stream) {
    if (!workspace) return SGL_ERR_INVALID_ARG;
    auto s = reinterpret_cast<cudaStream_t>(stream);
    int st = cuda_status(cudaStreamSynchronize(s));
    if (st) return st;
    uint32_t word = 0;
    st = cuda_status(cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost));
    if (st) return st;
    if (word == 0) return SGL_OK;
    st = cuda_status(cudaMemset(workspace, 0, sizeof(word)));
    if (st) return st;
    return SGL_ERR_BOUNDS;
}

}  // extern "C"
