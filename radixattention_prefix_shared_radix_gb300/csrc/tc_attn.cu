// Extend attention (bf16) on the 5th-generation tensor cores.
//
// "SGLang 深度拆解" (chenxutan.com/d/5669.html) §3.2 PagedPrefill and
// "SGLang 深度解读" section "5. Attention 层": the new tokens' K/V are in the
// pool before attention runs; new token i of request r attends to positions
// 0 .. prefix_len + i of its req_to_token row (the cached prefix plus the
// causal part of the new block).
//
// One CTA per pair of query tiles of 128 rows = (new token x query head of
// one KV head), 128/G new tokens per tile, consecutive tiles of one request;
// grid (pairs, KV heads).  The pair shares one K/V stream of 128-position
// blocks (2-stage rings for d = 128, 4 for d = 64, filled by a team of six
// gather warps) and runs the tcgen05 roles of tc_tile.cuh over positions
// 0 .. prefix_len + the pair's last new token, with the causal limit applied
// per row in the softmax.  480 threads (two softmax warpgroups, one MMA warp,
// six gather warps), ~193 KB of shared memory and all 512 TMEM columns: one
// CTA per SM, whose two query tiles take turns on the tensor core while each
// other's softmax runs.

#include <cudaTypedefs.h>

#include "tc_tile.cuh"

namespace sgl {
namespace {

using namespace sgldev;
using namespace tc;

// two query tiles, 128-position blocks (S MMAs of N = 128: an M = 128
// tcgen05 MMA costs about the same time for N = 64 as for N = 128), one score
// buffer each, 2 K/V stages (4 for d = 64), a gather team of 6 warps.  With
// an FP8 pool (codes staged by the gather team and converted to f16) one
// stage for d = 128, whose staging area takes the second stage's room.
template <int D, bool F8 = false>
using ExtCfg = TcCfg<D, false, 2, (F8 && D == 128) ? 1 : 2 * (128 / D), 6, 128, 1, F8>;

// Query tile pair (blockIdx.x, blockIdx.y) of the extend batch; false if empty.
__device__ bool extend_tile_info(const TcArgs& a, int* info) {
    const int tq = 128 / a.G;
    int acc_c = 0, acc_q = 0, req = -1, c0 = 0, qoff = 0;
    for (int r = 0; r < a.B; ++r) {
        const int e = __ldg(a.extend_lens + r);
        const int nt = e > 0 ? (e + tq - 1) / tq : 0;
        const int nc = (nt + 1) / 2;
        if ((int)blockIdx.x < acc_c + nc) {
            req = r;
            c0 = acc_c;
            qoff = acc_q;
            break;
        }
        acc_c += nc;
        acc_q += e > 0 ? e : 0;
    }
    if (req < 0) return false;
    const int pre = __ldg(a.prefix_lens + req), ext = __ldg(a.extend_lens + req);
    const int t0 = ((int)blockIdx.x - c0) * 2 * tq;
    const int na = min(tq, ext - t0), nb2 = min(tq, ext - t0 - tq);
    const int ntok = na + (nb2 > 0 ? nb2 : 0);
    if (pre < 0 || na <= 0 || (int64_t)pre + ext > a.ld || (int64_t)qoff + t0 + ntok > a.n_rows) {
        atomicOr(a.err, 2u);
        return false;
    }
    info[0] = req;                        // KV row
    info[1] = 0;                          // kv_begin
    info[2] = pre + t0 + ntok;            // kv_end
    info[3] = blockIdx.y;                 // KV head
    info[4] = na * a.G;                   // rows of tile 0
    info[5] = nb2 > 0 ? nb2 * a.G : 0;    // rows of tile 1 (0: absent)
    info[6] = qoff + t0;                  // first q row of tile 0
    info[7] = qoff + t0 + tq;             // first q row of tile 1
    info[8] = pre + t0;                   // causal limit of tile 0's first new token
    info[9] = pre + t0 + tq;              // causal limit of tile 1's first new token
    // fused KV write: positions from pre on are read from the new K/V, whose
    // row qoff holds position pre
    info[10] = a.kn != nullptr ? pre : INT_MAX;
    info[11] = qoff;
    return true;
}

template <int D, bool F8>
__global__ void __launch_bounds__(ExtCfg<D, F8>::kThreads, 1)
    extend_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tnk, const __grid_constant__ CUtensorMap tnv) {
    using C = ExtCfg<D, F8>;
    using Lay = typename C::Lay;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    int* info = reinterpret_cast<int*>(sm + Lay::OFF_INFO);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Lay::OFF_TMEM);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) info[15] = extend_tile_info(a, info) ? 1 : 0;
    __syncthreads();
    if (!info[15]) return;
    if (tid == 0) {
        tc_init_barriers<C>(smem_u32(sm + Lay::OFF_BAR));
        mbar_fence_init();
    }
    if (warp == C::kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(tslot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const TileInfo ti{info[0], info[1], info[2], info[3], {info[4], info[5]}, {info[6], info[7]}, {info[8], info[9]},
                      info[10], info[11]};
    TcState st{0u, 0u, false};
    tc_tile_run<C>(a, &tmk, &tmv, &tnk, &tnv, ti, sm, tbase, st, tid);
    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tbase));
    }
}

template <int D, bool F8>
constexpr int extend_smem() {
    return ExtCfg<D, F8>::Lay::END + 1024;   // + alignment slack
}
static_assert(extend_smem<128, false>() <= 232448 && extend_smem<64, false>() <= 232448 &&
                  extend_smem<128, true>() <= 232448 && extend_smem<64, true>() <= 232448,
              "shared memory per CTA");
static_assert(extend_smem<128, false>() > 116 * 1024 && extend_smem<64, false>() > 116 * 1024 &&
                  extend_smem<128, true>() > 116 * 1024 && extend_smem<64, true>() > 116 * 1024,
              "one CTA per SM: each allocates all 512 TMEM columns");

}  // namespace

namespace tc {

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 enc = [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            fn = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }();
    return enc;
}

int encode_rows_map(const void* base, int64_t rows, int D, CUtensorMap* m, int box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return (int)cudaErrorNotSupported;
    if (rows <= 0 || rows > (int64_t)INT32_MAX || box_rows < 1 || box_rows > 256) return (int)cudaErrorInvalidValue;
    const cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estride,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

int encode_pool_maps(const void* kp, const void* vp, int64_t num_slots, int Hkv, int D, CUtensorMap* mk,
                     CUtensorMap* mv) {
    struct Cache {
        const void *kp = nullptr, *vp = nullptr;
        int64_t ns = -1;
        int hkv = 0, d = 0;
        CUtensorMap mk, mv;
    };
    thread_local Cache c;
    if (c.kp != kp || c.vp != vp || c.ns != num_slots || c.hkv != Hkv || c.d != D) {
        const int64_t rows = num_slots * (int64_t)Hkv;
        c.kp = nullptr;
        if (const int e = encode_rows_map(kp, rows, D, &c.mk)) return e;
        if (const int e = encode_rows_map(vp, rows, D, &c.mv)) return e;
        c.kp = kp;
        c.vp = vp;
        c.ns = num_slots;
        c.hkv = Hkv;
        c.d = D;
    }
    *mk = c.mk;
    *mv = c.mv;
    return 0;
}

}  // namespace tc

// Extend over all requests: grid (pairs of query tiles of 128/G new tokens, KV heads).
template <int D, bool F8>
int launch_extend_tc(const void* q, const void* kp, const void* vp, const void* kn, const void* vn, void* kw, void* vw,
                     const int32_t* r2t, int64_t ld, const int32_t* pre, const int32_t* ext, int B, int64_t n_rows,
                     int64_t ctas, void* o, float* lse,
                     uint32_t* err, int Hq, int Hkv, int64_t num_slots, float scale_log2, float k_scale, float v_scale,
                     cudaStream_t s) {
    static const int attr = (int)cudaFuncSetAttribute(extend_tc_kernel<D, F8>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, extend_smem<D, F8>());
    if (attr) return attr;
    // the pools' TMA views (an FP8 pool's codes are copied with cp.async:
    // its maps stay zero and unused)
    CUtensorMap mk{}, mv{}, nk{}, nv{};
    if (!F8)
        if (const int e = tc::encode_pool_maps(kp, vp, num_slots, Hkv, D, &mk, &mv)) return e;
    if (kn) {
        if (const int e = tc::encode_rows_map(kn, n_rows * Hkv, D, &nk)) return e;
        if (const int e = tc::encode_rows_map(vn, n_rows * Hkv, D, &nv)) return e;
    }
    TcArgs a{};
    a.q = static_cast<const bf16*>(q);
    a.kp = static_cast<const bf16*>(kp);
    a.vp = static_cast<const bf16*>(vp);
    a.kn = static_cast<const bf16*>(kn);
    a.vn = static_cast<const bf16*>(vn);
    a.kw = static_cast<bf16*>(kw);
    a.vw = static_cast<bf16*>(vw);
    a.r2t = r2t;
    a.ld = ld;
    a.prefix_lens = pre;
    a.extend_lens = ext;
    a.B = B;
    a.n_rows = n_rows;
    a.o = static_cast<bf16*>(o);
    a.lse = lse;
    a.err = err;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.num_slots = num_slots;
    a.scale_log2 = scale_log2;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    extend_tc_kernel<D, F8><<<dim3((unsigned)ctas, (unsigned)Hkv), ExtCfg<D, F8>::kThreads, extend_smem<D, F8>(), s>>>(
        a, mk, mv, nk, nv);
    return (int)cudaGetLastError();
}

template int launch_extend_tc<64, false>(const void*, const void*, const void*, const void*, const void*, void*,
                                         void*, const int32_t*, int64_t, const int32_t*, const int32_t*, int,
                                         int64_t, int64_t, void*, float*, uint32_t*, int, int, int64_t, float,
                                         float, float, cudaStream_t);
template int launch_extend_tc<64, true>(const void*, const void*, const void*, const void*, const void*, void*,
                                         void*, const int32_t*, int64_t, const int32_t*, const int32_t*, int,
                                         int64_t, int64_t, void*, float*, uint32_t*, int, int, int64_t, float,
                                         float, float, cudaStream_t);
template int launch_extend_tc<128, false>(const void*, const void*, const void*, const void*, const void*, void*,
                                         void*, const int32_t*, int64_t, const int32_t*, const int32_t*, int,
                                         int64_t, int64_t, void*, float*, uint32_t*, int, int, int64_t, float,
                                         float, float, cudaStream_t);
template int launch_extend_tc<128, true>(const void*, const void*, const void*, const void*, const void*, void*,
                                         void*, const int32_t*, int64_t, const int32_t*, const int32_t*, int,
                                         int64_t, int64_t, void*, float*, uint32_t*, int, int, int64_t, float,
                                         float, float, cudaStream_t);

}  // namespace sgl
