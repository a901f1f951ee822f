// One decode step from host memory: the step's inputs go to the device in
// one copy, the decode runs, its outputs come back in one copy, all queued
// on the caller's stream by one call.
//
// The serving loop of the pages prepares a step's metadata on the CPU while
// the GPU runs the step before (CS349D lecture-16 notes §2.2, overlap
// scheduling; "SGLang 深度解读" section 2, Scheduler): each step then moves
// the new query rows, the grown req_to_token rows and the lengths to the
// device and reads the attention output back.  A loop that stages all of a
// step's inputs in one pinned buffer (and its outputs in another) makes one
// library call per step instead of one call per copy plus the decode.
#include <cuda_runtime.h>

#include "common.h"

namespace {
int status_of(cudaError_t e) {
    if (e == cudaSuccess) return SGL_OK;
    sgl::set_cuda_error(static_cast<int>(e));
    return SGL_ERR_CUDA;
}
}  // namespace

extern "C" int sgl_decode_step(const void* in_host, void* in_dev, size_t in_bytes, const void* q, const void* k_pool,
                               const void* v_pool, const int32_t* req_to_token, int64_t ld, const int32_t* seq_lens,
                               const sgl_plan* plan, void* o, float* lse, const void* out_dev, void* out_host,
                               size_t out_bytes, void* workspace, size_t ws_bytes, sgl_stream_t stream) {
    // every refusal before any GPU work
    if (in_bytes > 0 && (!in_host || !in_dev)) return SGL_ERR_INVALID_ARG;
    if (out_bytes > 0 && (!out_dev || !out_host)) return SGL_ERR_INVALID_ARG;
    if (const int st =
            sgl::decode_arg_status(plan, q, k_pool, v_pool, req_to_token, ld, seq_lens, o, lse, workspace, ws_bytes))
        return st;
    auto s = reinterpret_cast<cudaStream_t>(stream);
    if (in_bytes > 0) {
        const int st = status_of(cudaMemcpyAsync(in_dev, in_host, in_bytes, cudaMemcpyHostToDevice, s));
        if (st) return st;
    }
    if (const int st = sgl_decode_attn(q, k_pool, v_pool, req_to_token, ld, seq_lens, plan, o, lse, workspace,
                                       ws_bytes, stream))
        return st;
    if (out_bytes > 0)
        return status_of(cudaMemcpyAsync(out_host, out_dev, out_bytes, cudaMemcpyDeviceToHost, s));
    return SGL_OK;
}
