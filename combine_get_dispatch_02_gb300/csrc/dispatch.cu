// Dispatch kernels: scatter token rows into the receive rows of their top-k
// experts, as a BF16 bit copy or with the FP8 cast fused in.
//
// Operation: low_latency_dispatch of "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南"
// (section 核心API示例) with FP8 dispatch (section 核心优势; the DeepTech
// announcement of DeepEP, 010bt.com, lists native FP8 dispatch).  The FP8
// cast is per 128 channels: amax = max |x|, a = max(amax, 1e-4),
// scale = a / 448, q = e4m3(x * (448 / a)), nearest-even with saturation.
//
// Design: the work item is (token, 512-channel chunk) for one warp, 16
// channels (two 16-byte loads) per lane.  The token row is read once from
// HBM (read-only, no L1 allocation), cast once, and written K times with
// 16-byte streaming stores, so the kernel moves the algorithmic bytes and
// nothing else.  A 128-channel FP8 block is 8 lanes: its amax is three xor
// shuffles.  The kernel is launched with programmatic dependent launch behind
// the layout kernel: each warp loads and casts its first chunk before
// waiting for the slots.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 512;  // channels per warp item

__device__ __forceinline__ uint32_t cast_pair(float a, float b) {
    // two e4m3 codes, a in the low byte
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads) dispatch_kernel(const DispatchParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarp = ((int64_t)gridDim.x * kThreads) >> 5;
    const int H = p.H, K = p.K;
    const int nch = (H + kChunk - 1) / kChunk;
    const int64_t items = p.N * nch;
    bool waited = false;

    if (p.count_dst != nullptr && blockIdx.x == 0) {
        pdl_wait();
        waited = true;
        for (int e = threadIdx.x; e < p.E; e += kThreads) p.count_dst[e] = p.count_src[e];
    }

    const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(p.x);
    for (int64_t it = warp; it < items; it += nwarp) {
        const int64_t g = it / nch;
        const int c = (int)(it - g * nch) * kChunk + lane * 16;
        const bool act0 = c < H, act1 = c + 8 < H;
        const __nv_bfloat16 *xr = x + g * H + c;
        uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        if (act0) a = ld_nc_na_v4(xr);
        if (act1) b = ld_nc_na_v4(xr + 8);

        uint4 q = make_uint4(0, 0, 0, 0);
        float scale = 0.0f;
        if constexpr (FP8) {
            const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            float f[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                f[2 * j] = bf16_lo(u[j]);
                f[2 * j + 1] = bf16_hi(u[j]);
            }
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
            const float ac = fmaxf(amax, 1e-4f);
            scale = __fdiv_rn(ac, 448.0f);
            const float inv = __fdiv_rn(448.0f, ac);
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t lo = cast_pair(__fmul_rn(f[4 * j], inv), __fmul_rn(f[4 * j + 1], inv));
                const uint32_t hi = cast_pair(__fmul_rn(f[4 * j + 2], inv), __fmul_rn(f[4 * j + 3], inv));
                w[j] = lo | (hi << 16);
            }
            q = make_uint4(w[0], w[1], w[2], w[3]);
        }

        if (!waited) {
            pdl_wait();
            waited = true;
        }
        const int32_t my_slot = lane < K ? p.slot[g * K + lane] : -1;
        for (int k = 0; k < K; ++k) {
            const int32_t s = __shfl_sync(0xFFFFFFFFu, my_slot, k);
            if (s < 0 || !act0) continue;
            if constexpr (FP8) {
                uint8_t *dst = static_cast<uint8_t *>(p.recv) + (int64_t)s * H + c;
                st_cs_v4(dst, q);
                if ((lane & 7) == 0) p.recv_scales[(int64_t)s * (H / 128) + c / 128] = scale;
            } else {
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.recv) + (int64_t)s * H + c;
                st_cs_v4(dst, a);
                if (act1) st_cs_v4(dst + 8, b);
            }
        }
    }
}

template <bool FP8>
int blocks_per_sm() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dispatch_kernel<FP8>, kThreads, 0) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}

}  // namespace

int dispatch_blocks_per_sm(bool fp8) { return fp8 ? blocks_per_sm<true>() : blocks_per_sm<false>(); }

cudaError_t launch_dispatch(const DispatchParams &p, bool fp8, int max_blocks, bool pdl,
                            cudaStream_t stream) {
    const int nch = (p.H + kChunk - 1) / kChunk;
    const int64_t warps = p.N * nch;
    int64_t blocks = (warps + (kThreads / 32) - 1) / (kThreads / 32);
    if (blocks > max_blocks) blocks = max_blocks;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return fp8 ? cudaLaunchKernelEx(&cfg, dispatch_kernel<true>, p)
               : cudaLaunchKernelEx(&cfg, dispatch_kernel<false>, p);
}

}  // namespace ep
