// Row mover: the "wire" of a split (send / receive-hook) dispatch or combine.
//
// The hook-based overlap of "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南"
// (section 技术解析, 通信-计算重叠技术; the DeepTech announcement of DeepEP,
// 010bt.com, says the same) lets data move while the SMs compute, occupying no
// SM: the send call returns, a later hook call finishes the receive.  On one
// GPU the wire is this GPU's HBM and the engine that moves rows without SM
// work is the bulk-copy (TMA) unit: this kernel's threads only issue
// cp.async.bulk copies — global -> shared (completing on an mbarrier), then
// shared -> global to every destination row — so it can run on a few SMs
// while other kernels use the rest.
//
// One warp per CTA, a ring of `ring` row buffers: lane 0 keeps ring-1 row
// loads in flight; when a row has landed, lane k < K issues the copy to the
// k-th destination (one bulk group per lane and row), and the buffer is
// refilled once the copies of the row before it have read it.  Every
// mbarrier wait is bounded (about one second of %globaltimer, or the
// parameter's bound): on expiry the kernel sets kStatusTimeout in the status
// word, then waits, bounded again, for every load it issued that has not
// landed.  If one of those waits also gives up, a bulk load may still be
// writing into this CTA's shared memory after the kernel exits: the kernel
// sets kStatusInFlight as well (the device's later kernels cannot be trusted).
// Its own stores are drained before it returns.  A test can make the first
// wait run out without any load in flight: the item `withhold` is never
// loaded, so its barrier phase never completes.
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kMaxRing = 8;

__device__ __forceinline__ uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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
// Bounded wait (limit_ns of %globaltimer) for the phase with this parity;
// false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (!mbar_try(bar, parity))
        if (now_ns() - t0 > limit_ns) return false;
    return true;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__global__ void __launch_bounds__(32) move_rows_kernel(const MoveParams p) {
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t bars[kMaxRing];
    const int lane = threadIdx.x;
    const int NB = p.ring;
    const uint32_t rb = (uint32_t)p.row_bytes;
    const uint32_t sb = p.src_scales != nullptr ? (uint32_t)p.scale_bytes : 0u;
    const uint32_t buf = rb + sb;
    const int64_t G = gridDim.x;
    const int64_t cnt = p.n > (int64_t)blockIdx.x ? (p.n - 1 - blockIdx.x) / G + 1 : 0;
    const uint64_t limit = p.wait_ns > 0 ? (uint64_t)p.wait_ns : kMoveWaitNs;

    if (lane == 0) {
        for (int b = 0; b < NB; ++b) mbar_init(saddr(&bars[b]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    // the source rows (and slots) come from the kernels queued before
    pdl_wait();
    if (p.count_dst != nullptr && blockIdx.x == 0)
        for (int e = lane; e < p.E; e += 32) p.count_dst[e] = p.count_src[e];

    // source row of the CTA's i-th item, -1 for none
    auto src_row = [&](int64_t i) -> int64_t {
        const int64_t j = blockIdx.x + i * G;
        return p.gather ? (int64_t)p.slot[j] : j;
    };
    auto withheld = [&](int64_t i) { return blockIdx.x + i * G == p.withhold; };
    auto issue = [&](int64_t i) {  // lane 0
        const int b = (int)(i % NB);
        const uint32_t bar = saddr(&bars[b]);
        const int64_t s = src_row(i);
        if (withheld(i)) {
            // test hook: no load and no arrival, so this phase never completes
        } else if (s >= 0) {
            mbar_arrive_tx(bar, buf);
            bulk_load(saddr(ring + (size_t)b * buf), p.src + s * rb, rb, bar);
            if (sb) bulk_load(saddr(ring + (size_t)b * buf + rb), p.src_scales + s * sb, sb, bar);
        } else {
            mbar_arrive(bar);  // nothing to move: complete the phase
        }
    };

    int64_t issued = 0;
    if (lane == 0)
        for (; issued < NB - 1 && issued < cnt; ++issued) issue(issued);
    issued = __shfl_sync(0xFFFFFFFFu, issued, 0);

    bool ok = true;
    int64_t i = 0;
    for (; i < cnt; ++i) {
        const int b = (int)(i % NB);
        // every lane waits (the stores it issues read the landed row); the
        // outcome is made warp-uniform before anyone leaves the loop
        const bool landed = mbar_wait(saddr(&bars[b]), (uint32_t)((i / NB) & 1), limit);
        if (!__all_sync(0xFFFFFFFFu, landed)) {
            ok = false;
            break;
        }
        const int64_t j = blockIdx.x + i * G;
        const uint8_t *row = ring + (size_t)b * buf;
        if (lane < p.K) {
            int64_t d = -1;
            if (p.gather) {
                if (p.slot[j] >= 0) d = j;
            } else {
                d = p.slot[j * p.K + lane];
            }
            if (d >= 0) {
                bulk_store(p.dst + d * rb, saddr(row), rb);
                if (sb) bulk_store(p.dst_scales + d * sb, saddr(row + rb), sb);
            }
            bulk_commit();
            // the copies of the previous row have read its buffer
            bulk_wait_read_1();
        }
        __syncwarp();
        if (lane == 0 && issued < cnt) issue(issued);
        ++issued;
    }
    if (!ok) {
        // Loads issued for items i .. issued-1 (one per ring buffer, the item
        // that timed out included) land in this CTA's shared memory: wait for
        // each of them, bounded, before the CTA gives its shared memory up.
        // Every one is waited for, even after one wait gives up.
        bool drained = true;
        for (int64_t k = i; k < issued && k < cnt; ++k)
            if (!withheld(k) && !mbar_wait(saddr(&bars[k % NB]), (uint32_t)((k / NB) & 1), limit)) drained = false;
        if (lane == 0) atomicOr(p.status, drained ? kStatusTimeout : (kStatusTimeout | kStatusInFlight));
    }
    if (lane < p.K) bulk_wait_all();
}

// Reads a buffer larger than L2 so that the next kernel starts with an L2
// holding only clean lines of this buffer (the dirty lines of earlier kernels
// are written back here).  The loaded words feed a comparison that is never
// true in practice, so the loads are kept.
__global__ void l2_evict_kernel(const uint4 *p, int64_t n, uint32_t *sink) {
    uint32_t acc = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldcg(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (acc == 0x9E3779B9u && sink != nullptr) *sink = acc;
}

}  // namespace

cudaError_t launch_l2_evict(const void *buf, size_t bytes, int sms, cudaStream_t stream) {
    const int64_t n = (int64_t)(bytes / 16);
    if (n <= 0) return cudaSuccess;
    l2_evict_kernel<<<sms * 4, 512, 0, stream>>>(static_cast<const uint4 *>(buf), n, nullptr);
    return cudaGetLastError();
}

namespace {
int g_smem_sm = 0, g_smem_blk = 0, g_reserved = 0;
int g_static = 0;  // the kernel's static shared memory (the mbarriers)
}  // namespace

void move_init() {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&g_smem_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&g_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, move_rows_kernel) == cudaSuccess) g_static = (int)fa.sharedSizeBytes;
    // static + dynamic shared memory may not exceed the opt-in limit
    if (cudaFuncSetAttribute(move_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, g_smem_blk - g_static) !=
        cudaSuccess)
        g_smem_sm = 0;  // launches then report the failed set-up
    cudaGetLastError();
}

cudaError_t launch_move(MoveParams p, int sms, bool pdl, cudaStream_t stream) {
    const int smem_sm = g_smem_sm, smem_blk = g_smem_blk, reserved = g_reserved;
    if (smem_sm <= 0) return cudaErrorInitializationError;
    const size_t buf = (size_t)p.row_bytes + (p.src_scales != nullptr ? (size_t)p.scale_bytes : 0);
    // about 48 KB of ring per CTA (2..8 rows), as many CTAs per SM as fit (<= 8)
    int ring = (int)((48 << 10) / buf);
    ring = ring < 2 ? 2 : (ring > kMaxRing ? kMaxRing : ring);
    const size_t smem = (size_t)ring * buf;
    if (smem + g_static > (size_t)smem_blk) return cudaErrorInvalidConfiguration;
    int per_sm = (int)(smem_sm / (smem + reserved + g_static));
    per_sm = per_sm < 1 ? 1 : (per_sm > 8 ? 8 : per_sm);
    p.ring = ring;
    int64_t blocks = (int64_t)sms * per_sm;
    if (blocks > p.n) blocks = p.n;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, move_rows_kernel, p);
}

}  // namespace ep
