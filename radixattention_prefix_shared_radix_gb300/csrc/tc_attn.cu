// Extend attention (bf16) on the 5th-generation tensor cores.
//
// "SGLang 深度拆解" (chenxutan.com/d/5669.html) §3.2 PagedPrefill and
// "SGLang 深度解读" section "5. Attention 层": the new tokens' K/V are in the
// pool before attention runs; new token i of request r attends to positions
// 0 .. prefix_len + i of its req_to_token row (the cached prefix plus the
// causal part of the new block).
//
// One CTA per tile of 128 rows = (new token x query head of one KV head),
// 128/G new tokens of one request; grid (tiles, KV heads).  The tile runs the
// tcgen05 roles of tc_tile.cuh over positions 0 .. prefix_len + last new
// token of the tile, with the causal limit applied per row in the softmax.
// 224 threads, ~98 KB of shared memory and 256 TMEM columns per CTA, so two
// tiles share an SM and take turns on the tensor core and the softmax units.

#include "tc_tile.cuh"

namespace sgl {
namespace {

using namespace sgldev;
using namespace tc;

// Tile (blockIdx.x, blockIdx.y) of the extend batch; false if empty.
__device__ bool extend_tile_info(const TcArgs& a, int* info) {
    const int tq = 128 / a.G;
    int acc_t = 0, acc_q = 0, req = -1, tile0 = 0, qoff = 0;
    for (int r = 0; r < a.B; ++r) {
        const int e = __ldg(a.extend_lens + r);
        const int nt = e > 0 ? (e + tq - 1) / tq : 0;
        if ((int)blockIdx.x < acc_t + nt) {
            req = r;
            tile0 = acc_t;
            qoff = acc_q;
            break;
        }
        acc_t += nt;
        acc_q += e > 0 ? e : 0;
    }
    if (req < 0) return false;
    const int pre = __ldg(a.prefix_lens + req), ext = __ldg(a.extend_lens + req);
    const int t0 = ((int)blockIdx.x - tile0) * tq;
    const int ntok = min(tq, ext - t0);
    if (pre < 0 || ntok <= 0 || (int64_t)pre + ext > a.ld || (int64_t)qoff + t0 + ntok > a.n_rows) {
        atomicOr(a.err, 2u);
        return false;
    }
    info[0] = req;                // KV row
    info[1] = 0;                  // kv_begin
    info[2] = pre + t0 + ntok;    // kv_end
    info[3] = blockIdx.y;         // KV head
    info[4] = ntok * a.G;         // rows
    info[5] = qoff + t0;          // first q row
    info[6] = pre + t0;           // causal limit of the tile's first new token
    return true;
}

template <int D>
__global__ void __maxnreg__(128) extend_tc_kernel(const TcArgs a) {
    using Lay = TcLayout<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    int* info = reinterpret_cast<int*>(sm + Lay::OFF_INFO);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Lay::OFF_TMEM);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) info[7] = extend_tile_info(a, info) ? 1 : 0;
    __syncthreads();
    if (!info[7]) return;
    if (tid == 0) {
        tc_init_barriers<D, false>(smem_u32(sm + Lay::OFF_BAR));
        mbar_fence_init();
    }
    if (warp == 4) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;\n" ::"r"(smem_u32(tslot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const TileInfo ti{info[0], info[1], info[2], info[3], info[4], info[5], info[6]};
    TcState st{0u, 0u, false};
    tc_tile_run<D, false>(a, ti, sm, tbase, st, tid);
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;\n" ::"r"(tbase));
    }
}

template <int D>
constexpr int extend_smem() {
    return TcLayout<D>::END + 1024;   // + alignment slack
}

}  // namespace

// Extend over all requests: grid (tiles of 128/G new tokens, KV heads).
template <int D>
int launch_extend_tc(const void* q, const void* kp, const void* vp, const int32_t* r2t, int64_t ld,
                     const int32_t* pre, const int32_t* ext, int B, int64_t n_rows, int64_t tiles, void* o, float* lse,
                     uint32_t* err, int Hq, int Hkv, int64_t num_slots, float scale_log2, cudaStream_t s) {
    static const int attr = (int)cudaFuncSetAttribute(extend_tc_kernel<D>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, extend_smem<D>());
    if (attr) return attr;
    TcArgs a{};
    a.q = static_cast<const bf16*>(q);
    a.kp = static_cast<const bf16*>(kp);
    a.vp = static_cast<const bf16*>(vp);
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
    extend_tc_kernel<D><<<dim3((unsigned)tiles, (unsigned)Hkv), kTileThreads, extend_smem<D>(), s>>>(a);
    return (int)cudaGetLastError();
}

template int launch_extend_tc<64>(const void*, const void*, const void*, const int32_t*, int64_t, const int32_t*,
                                  const int32_t*, int, int64_t, int64_t, void*, float*, uint32_t*, int, int, int64_t,
                                  float, cudaStream_t);
template int launch_extend_tc<128>(const void*, const void*, const void*, const int32_t*, int64_t, const int32_t*,
                                   const int32_t*, int, int64_t, int64_t, void*, float*, uint32_t*, int, int, int64_t,
                                   float, cudaStream_t);

}  // namespace sgl
