// Identity expert: the stand-in for the expert computation between dispatch
// and combine in a round trip.  Every receive row that an entry of the token
// range received is written, as its expert's output, with the BF16 value the
// row stands for:
//   FP8 rows:  y[row, c] = bf16( e4m3(q[row, c]) * scale[row, c / 128] )
//              (the code is exact in fp32; one fp32 multiply and one
//              nearest-even bf16 rounding)
//   BF16 rows: y[row] = recv[row]  (bit copy)
// so that combine(identity(dispatch(x))) is the round trip of the FP8
// dispatch / BF16 combine pair of "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南"
// (section 核心优势).
//
// Design: the work item is (entry, 512-channel chunk) for one warp, taken
// 256 channels at a time: a lane converts 8 channels per pass, so each
// pass is one 8-byte code load (FP8) or 16-byte load (BF16) and one
// 16-byte store per lane, and a warp's store covers 512 contiguous bytes
// (whole 32-byte sectors; with 16 channels per lane each store instruction
// would half-fill 32 sectors, measured 16% slower).  A lane issues the
// item's two loads before the first conversion (items of 1024 or 2048
// channels, with more loads in flight, measured slower on a persistent
// grid).  Masked entries (no row) cost one slot load.  Reads
// bypass L1; the stores are ordinary so that, in a chunked round trip, the
// rows the combine reads next can still be in L2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kThreads = 256;
constexpr int kItem = 512;  // channels per warp item

// two e4m3 codes (low byte first) -> two floats, exactly (every e4m3 value
// is a half value)
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t pair) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(pair & 0xFFFFu), __NV_E4M3);
    return __half22float2(__half2(h));
}

__device__ __forceinline__ uint32_t bf16x2_rn(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads) expert_identity_kernel(const IdentityParams p) {
    constexpr int PASS = kItem / 256;  // 8 channels per lane and pass
    // the rows are written by the dispatch kernel queued just before
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarp = ((int64_t)gridDim.x * kThreads) >> 5;
    const int H = p.H;
    const int nch = (H + kItem - 1) / kItem;
    const int64_t items = p.n * nch;
    __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(p.y);

    for (int64_t it = warp; it < items; it += nwarp) {
        const int64_t i = it / nch;
        const int32_t s = p.slot[i];
        if (s < 0) continue;  // warp-uniform
        const int cb = (int)(it - i * nch) * kItem + lane * 8;
        uint4 v[PASS];  // FP8: 8 codes in .x/.y; BF16: 8 values
        float sc[PASS];
#pragma unroll
        for (int j = 0; j < PASS; ++j) {
            const int c = cb + j * 256;
            v[j] = make_uint4(0, 0, 0, 0);
            sc[j] = 0.0f;
            if (c < H) {
                if constexpr (FP8) {
                    const uint2 u = ld_nc_na_v2(static_cast<const uint8_t *>(p.recv) + (int64_t)s * H + c);
                    v[j].x = u.x;
                    v[j].y = u.y;
                    sc[j] = __ldg(p.recv_scales + (int64_t)s * (H / 128) + c / 128);
                } else {
                    v[j] = ld_nc_na_v4(static_cast<const __nv_bfloat16 *>(p.recv) + (int64_t)s * H + c);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < PASS; ++j) {
            const int c = cb + j * 256;
            if (c >= H) continue;
            uint4 o = v[j];
            if constexpr (FP8) {
                const float2 a = e4m3x2_to_float2(v[j].x), b = e4m3x2_to_float2(v[j].x >> 16);
                const float2 d = e4m3x2_to_float2(v[j].y), e = e4m3x2_to_float2(v[j].y >> 16);
                o.x = bf16x2_rn(__fmul_rn(a.x, sc[j]), __fmul_rn(a.y, sc[j]));
                o.y = bf16x2_rn(__fmul_rn(b.x, sc[j]), __fmul_rn(b.y, sc[j]));
                o.z = bf16x2_rn(__fmul_rn(d.x, sc[j]), __fmul_rn(d.y, sc[j]));
                o.w = bf16x2_rn(__fmul_rn(e.x, sc[j]), __fmul_rn(e.y, sc[j]));
            }
            *reinterpret_cast<uint4 *>(y + (int64_t)s * H + c) = o;
        }
    }
}

template <bool FP8>
int occupancy() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, expert_identity_kernel<FP8>, kThreads, 0) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}

}  // namespace

int identity_blocks_per_sm(bool fp8) { return fp8 ? occupancy<true>() : occupancy<false>(); }

cudaError_t launch_identity(const IdentityParams &p, bool fp8, int max_blocks, bool pdl, cudaStream_t stream) {
    const int nch = (p.H + kItem - 1) / kItem;
    const int64_t warps = p.n * nch;
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
    return fp8 ? cudaLaunchKernelEx(&cfg, expert_identity_kernel<true>, p)
               : cudaLaunchKernelEx(&cfg, expert_identity_kernel<false>, p);
}

}  // namespace ep
