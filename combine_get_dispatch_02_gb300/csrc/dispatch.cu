// Dispatch kernels: scatter token rows into the receive rows of their top-k
// experts, as a BF16 bit copy or with the FP8 cast fused in.
//
// Operation: low_latency_dispatch of "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南"
// (section 核心API示例) with FP8 dispatch (section 核心优势; the DeepTech
// announcement of DeepEP, 010bt.com, lists native FP8 dispatch).  The FP8
// cast is per 128 channels: amax = max |x|, a = max(amax, 1e-4),
// scale = a / 448, q = e4m3(x * (448 / a)), nearest-even with saturation.
//
// Three kernels.  Large dispatches (from 64K receive rows) run the token
// kernel: one CTA per token holds the row in registers and writes it to
// every receive row with 16-byte stores.  Otherwise, for hidden sizes that
// are a multiple of 512 (all the workloads), the row kernel stages a whole
// token row in shared memory and writes it with bulk asynchronous copies
// (producer warps and an issuer warp handing buffers over through
// mbarriers).  Otherwise the warp-item kernel does:
// the work item is (token, 512-channel chunk) for one warp, 16
// channels (two 16-byte loads) per lane.  The token row is read once from
// HBM (read-only, no L1 allocation), cast once, and written K times with
// 16-byte streaming stores, so the kernel moves the algorithmic bytes and
// nothing else.  A 128-channel FP8 block is 8 lanes: its amax is three xor
// shuffles.  The kernel is launched with programmatic dependent launch behind
// the layout kernel: each warp loads and casts its first chunk before
// waiting for the slots (x was written before the layout kernel started).
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

// Receive row of entry (g, lane), or -1 for none (lanes >= K).  Without a
// slot array token g goes to row g (K == 1).
__device__ __forceinline__ int32_t slot_of(const DispatchParams &p, int64_t g, int lane) {
    if (lane >= p.K) return -1;
    return p.slot != nullptr ? p.slot[g * p.K + lane] : (int32_t)g;
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

    if (!p.early_x && !waited) {  // x may be the output of the kernel just before
        pdl_wait();
        waited = true;
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
        const int32_t my_slot = slot_of(p, g, lane);
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

// ---------------------------------------------------------------- row kernel
// One CTA per token at a time.  H/16 producer threads (16 channels each) and
// one issuer warp.  The producers load the token row once (two tokens
// ahead), cast it once (FP8) and lay it out in a shared-memory row buffer;
// the issuer warp then has lane k < K copy the whole row (and its scale row)
// to the receive row of entry k with one bulk asynchronous copy
// (cp.async.bulk), so each destination row is one contiguous transfer by the
// copy engine.  NB row buffers form a ring with two mbarriers each:
//   full[b]   completes when every producer warp has written its part of the
//             buffer (one arrival per warp, after a proxy fence that makes
//             the writes visible to the copy engine);
//   empty[b]  completes when the copies of the buffer's row have read it
//             (the issuer's cp.async.bulk.wait_group.read, LAG tokens
//             later), so the producers may refill it.
// LAG < NB: the producers of token t wait for the release of token t - NB,
// which the issuer gives after token t - NB + LAG; with LAG >= NB that would
// be token t itself, which they have not written yet.
// No CTA-wide barrier per token: the producer warps run up to NB - LAG
// tokens ahead of the issuer and independently of one another.  Only the
// issuer waits for the layout kernel before it (programmatic dependent
// launch: it reads the slots); behind the library's own layout kernel the
// producers fill the ring meanwhile (x was written before that kernel
// started).  Every
// mbarrier wait is bounded (about one second); if one gives up the kernel
// sets kStatusTimeout, stops issuing, lets its copies finish and returns.
// Needs H % 512 == 0 and H/16 + 32 <= 1024 threads.
// CTAs per SM: about 1024 threads, at least 2 (measured best at H = 7168);
// FP8 rows at most 4 (H = 2048, top-6 / top-8: 0.90 of peak on 4 CTAs per SM
// against 0.77-0.85 on 8)
int row_blocks_per_sm(int H, bool fp8) {
    int b = 16384 / H;
    if (fp8 && b > 4) b = 4;
    return b < 2 ? 2 : (b > 16 ? 16 : b);
}

// tokens the issuer lets its copies run before it releases their buffer (< NB)
template <int NB>
struct Lag {
    static constexpr int value = NB > 2 ? 2 : 1;
};
constexpr uint64_t kRowWaitNs = 1000000000ull;     // bound of one mbarrier wait

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N committed groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait for the phase with this parity; false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (!mbar_try(bar, parity))
        if (now_ns() - t0 > kRowWaitNs) return false;
    return true;
}

// FP8 cast of this thread's 16 channels (two 16-byte bf16 loads): codes and
// the scale of their 128-channel block (8 lanes share a block).
__device__ __forceinline__ void cast16(uint4 ca, uint4 cb, uint4 &q, float &scale) {
    const uint32_t u[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
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

// This thread's part of a row buffer: FP8 codes + scale, or the bf16 copy.
template <bool FP8>
__device__ __forceinline__ void put_row(uint8_t *row, int t, int H, uint4 ca, uint4 cb, uint4 q, float scale) {
    if constexpr (FP8) {
        *reinterpret_cast<uint4 *>(row + t * 16) = q;
        if ((t & 7) == 0) reinterpret_cast<float *>(row + H)[t >> 3] = scale;
    } else {
        *reinterpret_cast<uint4 *>(row + t * 32) = ca;
        *reinterpret_cast<uint4 *>(row + t * 32 + 16) = cb;
    }
}

// ---------------------------------------------------------------- token kernel
// One CTA per token, a short-lived grid of N CTAs (or a persistent grid
// looping over the tokens when the SMs are limited).  H/16 threads: for FP8
// thread t holds channels [16t, 16t + 16) (two 16-byte loads) and casts them
// once (8 threads per 128-channel block, the amax by three xor shuffles);
// for BF16 thread t holds the row's 16-byte vectors t and t + H/16, so
// every store instruction of a warp writes 512 contiguous bytes.  The row
// then goes to the receive row of every top-k entry with plain 16-byte
// stores, one contiguous row written by the whole CTA within a few store
// instructions per warp.  Every CTA lets the next kernel launch as it
// starts (the dependents start once the last CTA has started); x may be
// read before the slots are waited for behind this library's own layout
// kernel (early_x).
template <bool FP8, int MINB>
__global__ void __launch_bounds__(MINB == 4 ? 512 : 1024, MINB) dispatch_token_kernel(const DispatchParams p) {
    pdl_launch_dependents();
    const int H = p.H, K = p.K, nt = H / 16;
    const int t = threadIdx.x, lane = t & 31;
    const bool act = t < nt;  // the block is rounded up to whole warps
    bool waited = false;
    if (p.count_dst != nullptr && blockIdx.x == 0) {
        pdl_wait();
        waited = true;
        for (int e = t; e < p.E; e += blockDim.x) p.count_dst[e] = p.count_src[e];
    }
    if (!p.early_x && !waited) {  // x may be the output of the kernel just before
        pdl_wait();
        waited = true;
    }
    const uint4 *x = static_cast<const uint4 *>(p.x);  // H / 8 vectors per row
    const int64_t nv = H / 8;
    const int i0 = FP8 ? 2 * t : t, i1 = FP8 ? 2 * t + 1 : t + nt;
    for (int64_t g = blockIdx.x; g < p.N; g += gridDim.x) {
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        if (act) {
            if constexpr (FP8) {  // 32 contiguous bytes per thread: the second load hits L1
                a = __ldg(x + g * nv + i0);
                b = __ldg(x + g * nv + i1);
            } else {  // each load instruction of a warp reads 512 contiguous bytes
                a = ld_nc_na_v4(x + g * nv + i0);
                b = ld_nc_na_v4(x + g * nv + i1);
            }
        }
        uint4 q = make_uint4(0, 0, 0, 0);
        float scale = 0.0f;
        if constexpr (FP8) cast16(a, b, q, scale);
        if (!waited) {
            pdl_wait();  // the slots of the layout kernel
            waited = true;
        }
        const int32_t my_slot = slot_of(p, g, lane);
        for (int k = 0; k < K; ++k) {
            const int32_t s = __shfl_sync(0xFFFFFFFFu, my_slot, k);
            if (s < 0 || !act) continue;
            if constexpr (FP8) {
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.recv) + (int64_t)s * H);
                dst[t] = q;
                if ((t & 7) == 0) p.recv_scales[(int64_t)s * (H / 128) + (t >> 3)] = scale;
            } else {
                uint4 *dst = static_cast<uint4 *>(p.recv) + (int64_t)s * nv;
                dst[i0] = a;
                dst[i1] = b;
            }
        }
    }
}

template <bool FP8, int NB>
__global__ void __launch_bounds__(1024, 1) dispatch_row_kernel(const DispatchParams p) {
    extern __shared__ __align__(128) uint8_t row_smem[];
    __shared__ __align__(8) uint64_t full[NB], empty[NB];
    const int H = p.H, K = p.K;
    const int t = threadIdx.x, lane = t & 31;
    const int np = H / 16;                      // producer threads; the issuer warp follows them
    const int rowb = FP8 ? H + H / 32 : 2 * H;  // bytes of one buffer
    const int64_t G = gridDim.x;
    if (t == 0) {
        for (int b = 0; b < NB; ++b) {
            mbar_init(smem_addr(&full[b]), (uint32_t)(np / 32));
            mbar_init(smem_addr(&empty[b]), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (t >= np) {
        // ------------------------------------------------ issuer warp
        pdl_wait();  // slots (and counts) of the layout kernel
        if (p.count_dst != nullptr && blockIdx.x == 0)
            for (int e = lane; e < p.E; e += 32) p.count_dst[e] = p.count_src[e];
        const int payload = FP8 ? H : 2 * H;
        int64_t g = blockIdx.x;
        int32_t s0 = g < p.N ? slot_of(p, g, lane) : -1;          // this token's slots,
        int32_t s1 = g + G < p.N ? slot_of(p, g + G, lane) : -1;  // and the next one's
        bool ok = true;
        for (int it = 0; g < p.N; ++it, g += G) {
            const int b = it % NB;
            const int32_t my_slot = s0;
            s0 = s1;
            s1 = g + 2 * G < p.N ? slot_of(p, g + 2 * G, lane) : -1;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&full[b]), (uint32_t)((it / NB) & 1)))) {
                ok = false;
                break;
            }
            const uint8_t *row = row_smem + b * rowb;
            if (lane < K) {
                if (my_slot >= 0) {
                    bulk_store(static_cast<uint8_t *>(p.recv) + (int64_t)my_slot * payload, smem_addr(row), payload);
                    if constexpr (FP8)
                        bulk_store(p.recv_scales + (int64_t)my_slot * (H / 128), smem_addr(row + H), H / 32);
                }
                bulk_commit();
                bulk_wait_read<Lag<NB>::value>();  // the copies of token it - LAG have read their buffer
            }
            __syncwarp();
            if (lane == 0 && it >= Lag<NB>::value) mbar_arrive(smem_addr(&empty[(it - Lag<NB>::value) % NB]));
        }
        if (!ok && lane == 0 && p.status != nullptr) atomicOr(p.status, kStatusTimeout);
        // every copy of this CTA is issued: the kernel queued behind (e.g. the
        // combine) may start its CTAs now; its griddepcontrol.wait still
        // waits for this grid to complete and its writes to be visible
        pdl_launch_dependents();
        if (lane < K) bulk_wait_all();  // copies read shared memory until they finish
        return;
    }

    // ---------------------------------------------------- producer warps
    if (!p.early_x) pdl_wait();  // x may be the output of the kernel just before
    const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(p.x);
    int64_t g = blockIdx.x;
    uint4 a = make_uint4(0, 0, 0, 0), b = a, a2 = a, b2 = a;
    if (g < p.N) {
        a = ld_nc_na_v4(x + g * H + t * 16);
        b = ld_nc_na_v4(x + g * H + t * 16 + 8);
    }
    if (g + G < p.N) {
        a2 = ld_nc_na_v4(x + (g + G) * H + t * 16);
        b2 = ld_nc_na_v4(x + (g + G) * H + t * 16 + 8);
    }
    for (int it = 0; g < p.N; ++it, g += G) {
        const uint4 ca = a, cb = b;
        a = a2;
        b = b2;
        if (g + 2 * G < p.N) {
            a2 = ld_nc_na_v4(x + (g + 2 * G) * H + t * 16);
            b2 = ld_nc_na_v4(x + (g + 2 * G) * H + t * 16 + 8);
        }
        uint4 q = make_uint4(0, 0, 0, 0);
        float scale = 0.0f;
        if constexpr (FP8) cast16(ca, cb, q, scale);
        const int buf = it % NB;
        // the buffer's previous row (NB tokens ago) must have been read
        if (it >= NB && !__all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&empty[buf]), (uint32_t)((it / NB - 1) & 1)))) {
            if (lane == 0 && p.status != nullptr) atomicOr(p.status, kStatusTimeout);
            return;
        }
        put_row<FP8>(row_smem + buf * rowb, t, H, ca, cb, q, scale);
        fence_proxy_async_smem();  // make the writes visible to the copy engine
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&full[buf]));
    }
}

bool row_kernel_fits(int H) { return H % 512 == 0 && H / 16 + 32 <= 1024; }

}  // namespace

bool token_kernel_fits(int H, bool fp8) { return H % (fp8 ? 128 : 16) == 0 && H / 16 <= 1024; }

// Measured over the sweep grid (T >= 32 tokens per rank, R in {8, 32}, H in
// {2048, 4096, 7168}, top-2/6/8, BF16 and FP8, cached layout): from 64K
// receive rows the token kernel takes 0.79-0.98 of the row kernel's time
// (FP8 at top-2 and H = 7168: 1.00-1.02); at 32K rows and below it ties or
// loses (the low-latency size, where the row kernel's ring also overlaps
// more of the layout kernel before it).
bool token_kernel_rule(int64_t N, int K, int H, bool fp8, bool sm_limited) {
    return !sm_limited && token_kernel_fits(H, fp8) && N * K >= 65536;
}

namespace {

size_t row_smem_bytes(bool fp8, int H) { return 2 * (size_t)(fp8 ? H + H / 32 : 2 * H); }

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

int dispatch_row_ctas_rule(int H, bool fp8) { return row_blocks_per_sm(H, fp8); }

int dispatch_blocks_per_sm(bool fp8) { return fp8 ? blocks_per_sm<true>() : blocks_per_sm<false>(); }

namespace {
int g_smem_per_sm = 0;        // shared memory per SM
int g_smem_reserved = 0;      // shared memory the system reserves per CTA
int g_smem_per_block = 0;     // largest dynamic shared memory of one CTA

// Dynamic shared memory that lets at most `blocks` CTAs of the row kernel
// share an SM.  The grid is persistent with a fixed share of tokens per CTA,
// so the CTAs must spread evenly: when the kernel starts early behind the
// layout kernel (programmatic dependent launch) the scheduler would
// otherwise pack extra CTAs onto the free SMs and those SMs would finish
// last.
size_t row_smem_for_occupancy(bool fp8, int H, int blocks) {
    const size_t need = row_smem_bytes(fp8, H);
    if (g_smem_per_sm <= 0) return need;
    const int64_t cap = (int64_t)g_smem_per_sm / (blocks + 1) - g_smem_reserved + 16;  // (static: 16 * NB bytes)
    size_t s = cap > (int64_t)need ? (size_t)cap : need;
    s = (s + 15) / 16 * 16;
    return s > (size_t)g_smem_per_block ? need : s;
}
}  // namespace

namespace {
// The most dynamic shared memory a kernel may ask for: the opt-in limit less
// its static shared memory (the row kernel's mbarriers).
template <typename F>
void allow_smem(F kernel) {
    cudaFuncAttributes fa;
    const int st = cudaFuncGetAttributes(&fa, kernel) == cudaSuccess ? (int)fa.sharedSizeBytes : 1024;
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, g_smem_per_block - st);
}
}  // namespace

void dispatch_init() {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&g_smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    cudaDeviceGetAttribute(&g_smem_per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    // the row kernel asks for more than the 48 KB default (see above)
    allow_smem(dispatch_row_kernel<false, 2>);
    allow_smem(dispatch_row_kernel<false, 4>);
    allow_smem(dispatch_row_kernel<false, 6>);
    allow_smem(dispatch_row_kernel<false, 8>);
    allow_smem(dispatch_row_kernel<true, 2>);
    allow_smem(dispatch_row_kernel<true, 4>);
    allow_smem(dispatch_row_kernel<true, 6>);
    allow_smem(dispatch_row_kernel<true, 8>);
    cudaGetLastError();
}

namespace {
// Row buffers in the ring and the dynamic shared memory of one CTA: the
// size that keeps a further row CTA off the SM (row_smem_for_occupancy),
// and as many buffers (8, 6, 4 or 2) as fit in it.  The share of the SM this
// leaves free is where the next kernel's CTAs start while the dispatch ends
// (it lets them launch early): a ring sized to the whole share (8 BF16 rows
// of 14 KB) left no room for them, and the BF16 step behind it took 1575
// instead of 1338 us at 8 x 4096 tokens, for no gain in the dispatch itself.
void row_ring(bool fp8, int H, int blocks, int *nb, size_t *smem) {
    const size_t rowb = fp8 ? (size_t)H + H / 32 : 2 * (size_t)H;
    const size_t cap = row_smem_for_occupancy(fp8, H, blocks);
    const size_t fit = cap / rowb;
    *nb = fit >= 8 ? 8 : (fit >= 6 ? 6 : (fit >= 4 ? 4 : 2));
    *smem = cap;  // >= 2 rows
}

template <bool FP8>
cudaError_t launch_row(const cudaLaunchConfig_t &cfg, int nb, const DispatchParams &p) {
    switch (nb) {
        case 8: return cudaLaunchKernelEx(&cfg, dispatch_row_kernel<FP8, 8>, p);
        case 6: return cudaLaunchKernelEx(&cfg, dispatch_row_kernel<FP8, 6>, p);
        case 4: return cudaLaunchKernelEx(&cfg, dispatch_row_kernel<FP8, 4>, p);
        default: return cudaLaunchKernelEx(&cfg, dispatch_row_kernel<FP8, 2>, p);
    }
}
}  // namespace

cudaError_t launch_dispatch(const DispatchParams &p, bool fp8, int max_blocks, bool pdl,
                            cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (p.token_grid > 0 && token_kernel_fits(p.H, fp8)) {
        int64_t blocks = p.N < p.token_grid ? p.N : p.token_grid;
        if (blocks < 1) blocks = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks, 1, 1);
        cfg.blockDim = dim3((unsigned)((p.H / 16 + 31) / 32 * 32), 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        // FP8 rows of up to 512 threads: registers for 4 CTAs per SM (3 otherwise)
        if (fp8 && cfg.blockDim.x <= 512) return cudaLaunchKernelEx(&cfg, dispatch_token_kernel<true, 4>, p);
        return fp8 ? cudaLaunchKernelEx(&cfg, dispatch_token_kernel<true, 1>, p)
                   : cudaLaunchKernelEx(&cfg, dispatch_token_kernel<false, 1>, p);
    }
    if (row_kernel_fits(p.H) && p.row_sms > 0) {
        const int bps = p.row_bps > 0 ? p.row_bps : row_blocks_per_sm(p.H, fp8);
        int64_t blocks = (int64_t)p.row_sms * bps;
        if (blocks > p.N) blocks = p.N;
        if (blocks < 1) blocks = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks, 1, 1);
        cfg.blockDim = dim3(p.H / 16 + 32, 1, 1);
        int nb = 2;
        size_t smem = 0;
        row_ring(fp8, p.H, bps, &nb, &smem);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        return fp8 ? launch_row<true>(cfg, nb, p) : launch_row<false>(cfg, nb, p);
    }
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
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return fp8 ? cudaLaunchKernelEx(&cfg, dispatch_kernel<true>, p)
               : cudaLaunchKernelEx(&cfg, dispatch_kernel<false>, p);
}

}  // namespace ep
