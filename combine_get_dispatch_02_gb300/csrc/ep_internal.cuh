// Internal declarations shared by the libep translation units: kernel
// parameter blocks, launchers and small device helpers.  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ep {

// Bits of the per-context device status word.
constexpr uint32_t kStatusBadExpert = 1u;  // topk_idx entry outside [-1, E)
constexpr uint32_t kStatusCapacity = 2u;   // padded expert buffer offered > R*Tmax entries
constexpr uint32_t kStatusTimeout = 4u;    // a bounded wait of a copy kernel gave up
constexpr uint32_t kStatusInFlight = 8u;   // ... and its loads may still land in freed shared memory

constexpr int kLayoutPadded = 0;
constexpr int kLayoutPacked = 1;

// ------------------------------------------------------------------ layout
struct LayoutParams {
    const int64_t *topk_idx;   // [N*K]
    int32_t R, T, K, E, L;     // E = keys (experts, or ranks in rank mode); L = experts per rank
    int32_t num_experts;       // valid ids are [0, num_experts)
    int32_t rank_mode;         // 1: keys are destination ranks, one entry per (token, rank)
    const float *topk_weights; // [N*K] or nullptr (rank mode: weights of the received rows)
    int32_t *recv_topk_idx;    // rank mode: [rows*K] local expert ids or -1, or nullptr
    float *recv_topk_weights;  // rank mode: [rows*K] or nullptr
    int32_t layout;
    int64_t N;                 // R*T
    int64_t cap;               // rows per expert buffer (padded) or N*K (packed)
    int32_t *slot;             // [N*K]
    int32_t *src_info;         // [rows]
    int32_t *cnt_er;           // [E*R]
    int32_t *off_er;           // [E*R]
    int64_t *base;             // [E]
    int32_t *tokens_per_expert;       // [E] (handle)
    int32_t *user_tokens_per_expert;  // [E] or nullptr
    int32_t *tokens_per_rank;         // [R] or nullptr
    uint8_t *is_token_in_rank;        // [N*R] or nullptr
    uint32_t *status;
    int32_t staged;            // set by launch_layout: entries staged in shared memory
    int32_t er_span;           // set by launch_layout: ranks per CTA for the (e, r) counts
    // grid form (launch_layout_grid): per-CTA key totals -> prefixes [grid_ctas][E]
    int32_t *cta_hist;
    uint32_t *grid_bar;           // grid form: barrier counter (zero between launches; each launch
                                  // puts it back to zero as its last CTA leaves)
    int32_t grid_ctas, grid_tpc;  // set by launch_layout_grid: CTAs, tokens per CTA
};

// Launch the single-cluster layout kernel.  cluster_size / threads come from
// layout_pick_shape.  Returns the launch error.
cudaError_t launch_layout(const LayoutParams &p, int cluster_size, int threads,
                          cudaStream_t stream);
// Dynamic shared memory the layout kernel needs for these sizes.
size_t layout_smem_bytes(int E, int R, int threads, int cluster_size);
// Largest cluster size (16, 8, 4, 2 or 1) and thread count the device can run
// for these sizes (1024 threads first when many_entries); false if none fits.
bool layout_pick_shape(int E, int R, int *cluster_size, int *threads, bool many_entries = false);
// Entries (R*T*K) from which the many-entries shape is used.
constexpr int64_t kLayoutManyEntries = 65536;
// The same layout from one cooperative kernel over `ctas` CTAs (count, scan,
// write, between grid barriers), for many entries: the single cluster leaves
// most SMs idle.  Needs p.cta_hist with ctas * E ints and p.grid_bar (zero
// before the first launch).  Zeroes tokens_per_rank and cnt_er itself; no
// host-side copy precedes it.  ctas <= 512.
cudaError_t launch_layout_grid(LayoutParams p, int ctas, cudaStream_t stream);
// Entries from which the grid form is used (measured crossovers of the time
// layout + dispatch adds to dispatch alone: expert layout 32K / 64K entries
// cluster ahead by 9 / 3-5 us, 256K grid ahead by 14 us; rank layout grid
// ahead from 48K entries, tied at 32K; below them the single cluster wins
// because it has no grid barriers and no zeroing copies, and the dispatch
// casts rows on the SMs it leaves free).
constexpr int64_t kLayoutGridEntries = 131072;
constexpr int64_t kLayoutGridEntriesRank = 49152;

// ------------------------------------------------------------------ dispatch
struct DispatchParams {
    const void *x;             // bf16 [N, H]
    const int32_t *slot;       // [N*K]
    void *recv;                // bf16 or e4m3 [rows, H]
    float *recv_scales;        // [rows, H/128] (FP8)
    int64_t N;
    int32_t K, H;
    const int32_t *count_src;  // [E] copied to count_dst by block 0, or nullptr
    int32_t *count_dst;
    int32_t E;
    int32_t row_sms;           // SMs for the row kernel (H % 512 == 0), 0 = use the warp-item kernel
    // slot == nullptr: token g goes to row g (K must be 1): the send buffer of a split dispatch
    int32_t row_bps;           // row kernel CTAs per SM, 0 = the built-in rule (from H)
    uint32_t *status;          // row kernel: kStatusTimeout if one of its bounded waits gave up
    int32_t early_x;           // 1: the kernel is launched behind this library's layout kernel(s),
                               // which started after x was written, so x may be read before
                               // griddepcontrol.wait; 0: wait first (x may come from the kernel
                               // just before)
    int64_t token_grid;        // > 0: the token kernel (one CTA per token) on at most this many
                               // CTAs; 0: the row or the warp-item kernel (row_sms)
};

cudaError_t launch_dispatch(const DispatchParams &p, bool fp8, int max_blocks,
                            bool pdl, cudaStream_t stream);
// Whether the token kernel runs this hidden size (H % 16 == 0, H / 16 <= 1024;
// FP8: H % 128 == 0).
bool token_kernel_fits(int H, bool fp8);
// The built-in rule's choice of the token kernel for N tokens of K entries
// (large dispatches on all SMs).
bool token_kernel_rule(int64_t N, int K, int H, bool fp8, bool sm_limited);
// The row dispatch kernel's CTAs per SM by the built-in rule (from H and the payload).
int dispatch_row_ctas_rule(int H, bool fp8);
// Resident blocks per SM of the warp-item dispatch kernel (for grid sizing).
int dispatch_blocks_per_sm(bool fp8);
// One-time kernel attribute set-up (call with the device current).
void dispatch_init();

// ------------------------------------------------------------------ combine
struct CombineParams {
    const void *y;             // bf16 [rows, H]
    const float *weights;      // [N*K] or nullptr (all ones)
    const int32_t *slot;       // [N*K]
    void *out;                 // bf16 [N, H]
    int64_t N;
    int32_t K, H;
    int32_t max_valid;         // most entries of one token that have rows (K, or min(K, R) by rank)
    int32_t token_major;       // 1: entry (g, k) with slot >= 0 reads row g*K + k of y (a staging
                               // buffer in token order) instead of row slot
    int32_t cpi;               // 256-channel chunks per work item (1, 2, 4), 0 = the rule (from max_valid)
};

cudaError_t launch_combine(const CombineParams &p, int max_blocks, bool pdl,
                           cudaStream_t stream);
// The combine's chunks per work item by the built-in rule (from the most
// entries a token can have rows for).
int combine_cpi_rule(int max_valid);
// Resident combine CTAs per SM for the chunks per item that max_valid (or a
// nonzero cpi) selects.
int combine_blocks_per_sm(int max_valid, int cpi = 0);

// ------------------------------------------------------------------ row mover (copy engine)
// Moves rows with bulk asynchronous copies only (global -> shared ->
// global); the SM threads just issue them.
//   fan-out (gather == 0): item g = source row g, copied to the rows
//            slot[g*K + k] >= 0 of dst (the receive half of a split dispatch)
//   gather  (gather == 1): item i = entry, row slot[i] >= 0 of src copied to
//            row i of dst, K = 1 (the send half of a split combine)
// Each row is row_bytes (+ scale_bytes of scales when scales are given).
struct MoveParams {
    const uint8_t *src;
    const uint8_t *src_scales;  // or nullptr
    uint8_t *dst;
    uint8_t *dst_scales;
    const int32_t *slot;
    int64_t n;                  // items
    int32_t K;
    int32_t gather;
    int32_t row_bytes, scale_bytes;   // multiples of 16
    int32_t ring;               // buffers per CTA (2..8), set by launch_move
    const int32_t *count_src;   // [E] copied to count_dst by block 0, or nullptr
    int32_t *count_dst;
    int32_t E;
    uint32_t *status;
    int64_t withhold;           // test hook: item whose load is never issued (-1: none)
    int64_t wait_ns;            // bound of each mbarrier wait, 0 = kMoveWaitNs
};
constexpr uint64_t kMoveWaitNs = 1000000000ull;  // one second

// Launch on `sms` SMs (as many CTAs per SM as shared memory allows).
cudaError_t launch_move(MoveParams p, int sms, bool pdl, cudaStream_t stream);
// One-time set-up with the device current (shared memory limits).
void move_init();
// Read `bytes` (> L2) of `buf`: afterwards L2 holds only clean lines.
cudaError_t launch_l2_evict(const void *buf, size_t bytes, int sms, cudaStream_t stream);

// ------------------------------------------------------------------ rank runs
// Send rows of the rank-deduplicated transport (source-major runs; see
// rank_transport.cu).  R <= kRankRunsMaxRanks.
constexpr int kRankRunsMaxRanks = 32;
struct RankSendParams {
    const int64_t *topk_idx;   // [N*K]
    const int32_t *slot;       // [N*K] receive rows of the rank layout
    const int32_t *cnt_er;     // [R*R] cnt_er[d*R + r]: tokens source r carries to d
    const int32_t *off_er;     // [R*R] first row of (d, r) relative to base[d]
    const int64_t *base;       // [R]
    int32_t *send_slot;        // [N*K] out
    int64_t N;
    int32_t R, T, K, L;
};
cudaError_t launch_rank_send_slots(const RankSendParams &p, int sms, cudaStream_t stream);

// ------------------------------------------------------------------ identity expert
struct IdentityParams {
    const void *recv;          // e4m3 or bf16 [rows, H]
    const float *recv_scales;  // [rows, H/128] (FP8)
    const int32_t *slot;       // the range's entries [n]
    int64_t n;
    int32_t H;
    void *y;                   // bf16 [rows, H]
};

cudaError_t launch_identity(const IdentityParams &p, bool fp8, int max_blocks, bool pdl,
                            cudaStream_t stream);
int identity_blocks_per_sm(bool fp8);

// ------------------------------------------------------------------ device helpers
#ifdef __CUDACC__
// Programmatic dependent launch: let the next kernel in the stream start, and
// wait for the previous one's results.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// 16-byte read-only load that does not allocate in L1 (the buffer is not
// written while the kernel runs).
__device__ __forceinline__ uint4 ld_nc_na_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 8-byte form of the load above.
__device__ __forceinline__ uint2 ld_nc_na_v2(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// 16-byte streaming store (evict-first): the written rows are not read again
// by this kernel.
__device__ __forceinline__ void st_cs_v4(void *p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// bf16 pair (low half = first element) -> two floats, exactly.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
#endif

}  // namespace ep
