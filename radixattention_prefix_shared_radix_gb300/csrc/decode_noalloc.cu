// Decode attention for callers that cannot allocate device memory.
//
// sgl_decode_attn needs a caller-allocated workspace (plan tables, the fp32
// partial results of the split-KV work items, merge counters, error word).
// Some callers cannot provide one: a serving loop whose device memory is
// owned by another allocator and has a fixed budget that must not grow, or
// a latency-critical path that must avoid cudaMalloc because it can
// synchronize the device.  This entry point uses a fixed scratch array that
// lives in the library's own device image instead, so it allocates nothing
// per call.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds it until the process exits.  Host code cannot use the
// array's name as a device address, so the address is looked up once per
// device with cudaGetSymbolAddress (on the first call made on that device,
// with that device current) and cached; a device reset is not supported
// (the cached address would be stale afterwards).

#include <cuda_runtime.h>

#include <mutex>

#include "common.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(64) << 20;   // 64 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" int sgl_decode_attn_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* req_to_token, int64_t ld, const int32_t* seq_lens,
                                       const sgl_plan* plan, void* o, float* lse, sgl_stream_t stream) {
    // every refusal happens here, before the plan upload below writes to
    // the shared scratch: the scratch size, then the same argument checks
    // as sgl_decode_attn
    if (!plan || plan->kind != 0) return SGL_ERR_INVALID_ARG;
    sgl_plan_info_t info;
    int st = sgl_plan_info(plan, &info);
    if (st) return st;
    if (info.workspace_bytes < 0 || (size_t)info.workspace_bytes > kNoallocScratchBytes) return SGL_ERR_WORKSPACE;
    const int32_t B = plan->params.batch;
    if (B > 0 && (!q || !o || !lse || !seq_lens)) return SGL_ERR_INVALID_ARG;
    if (plan->n_items > 0 && (!k_pool || !v_pool || !req_to_token || ld < plan->max_pos)) return SGL_ERR_INVALID_ARG;
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al16(q) || !al16(k_pool) || !al16(v_pool) || !al16(o)) return SGL_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        sgl::set_cuda_error((int)e);
        return SGL_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SGL_ERR_UNSUPPORTED;
    void* ptr = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_addr[dev]) {
            void* addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_decode_scratch);
            if (e != cudaSuccess || !addr) {
                sgl::set_cuda_error((int)e);
                return SGL_ERR_CUDA;
            }
            g_scratch_addr[dev] = addr;
        }
        ptr = g_scratch_addr[dev];
    }
    // rewrites the plan tables, clears the error word and the merge counters
    st = sgl_plan_upload(plan, ptr, kNoallocScratchBytes, stream);
    if (st) return st;
    return sgl_decode_attn(q, k_pool, v_pool, req_to_token, ld, seq_lens, plan, o, lse, ptr, kNoallocScratchBytes,
                           stream);
}
