// reduce_apply.cu -- W-way aggregation of the workers' wire words, the
// global sign, and the parameter update.
//
// "Lion Cub: Minimizing Communication Overhead in Distributed Lion", "What
// carries the argument": the workers exchange a quantized sum of their update
// vectors, after which a global sign is taken.  In sign mode the sum of the
// +-1 votes is 2*popcount - W (majority vote; "Communication Efficient
// Distributed Training with Distributed Lion", "Approach", also gives the
// average agg/W); in L1 mode it is the integer sum of the Eq. (1) codes.
// theta then takes the textbook Lion step with decoupled weight decay.
//
// One thread per 8 consecutive elements.  Sign mode: the thread reads one
// byte of every worker's words (its 8 bits) and counts set bits per element
// with byte-lane counters -- each nibble is spread to four byte lanes by one
// multiply (bit j of the nibble lands on bit 8j), so one 32-bit add counts
// four elements at once (exact for W <= 255).  L1 mode: the thread reads
// 8*n bits per worker and sign-extends each field.  Both read theta with
// 16-byte loads and write it back once.
#include "aggregate.cuh"

namespace lc {
namespace {

template <int NB>
__global__ void __launch_bounds__(256) k_reduce_apply(const StepArgs a)
{
    __shared__ float avg_tab[kAvgTab];
    fill_avg_table(a, avg_tab);
    __syncthreads();
    const int64_t e0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kVec;
    if (e0 >= a.d)
        return;
    const int valid = (a.d - e0 >= kVec) ? kVec : static_cast<int>(a.d - e0);
    if (!in_bounds(a, (e0 * NB) / 32 + (kVec * NB + 31) / 32 <= a.wire_stride))
        return;
    int agg[kVec];
    aggregate8<NB>(a, e0, agg);
    float th[kVec];
    load_f32(a.theta, e0, valid, th);
#pragma unroll
    for (int j = 0; j < kVec; ++j)
        th[j] = lion_apply(th[j], direction(a, agg[j], avg_tab), a.lr, a.wd);
    store_f32(a.theta, e0, valid, th);
}

// ---- staged variant: the block's wire bytes arrive by bulk copy ------------
//
// One thread issues, per worker, one cp.async.bulk of the bytes that cover
// the block's elements (16-byte aligned: the block's byte offset is a
// multiple of 256*NB and every worker's row is padded to 16 bytes) into
// shared memory, completing on one mbarrier; meanwhile every thread loads its
// theta.  The wait is bounded: if the copies have not landed after
// kWaitLimit polls the block records an error in a.status, waits once more
// (bounded the same way) for its copies to land, so that none is still
// writing to the block's shared memory when it is released, and returns.

constexpr uint32_t kWaitLimit = 1u << 20;
// Element groups of 2048 per block (one group of 8 per thread each): the
// block's fixed cost -- barrier set-up, copy issue, the wait -- is paid once
// per kStagedGroups * 2048 elements.
constexpr int kStagedGroups = 2;

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Polls the mbarrier at shared address b until phase 0 completes, at most
// kWaitLimit times; true when it completed.
__device__ __forceinline__ bool wait_phase0(uint32_t b)
{
    uint32_t ok = 0;
    for (uint32_t it = 0; it < kWaitLimit && !ok; ++it)
        asm volatile("{\n .reg .pred P;\n mbarrier.try_wait.parity.shared::cta.b64 P, [%1], 0;\n selp.u32 %0, 1, 0, P;\n}"
                     : "=r"(ok) : "r"(b) : "memory");
    return ok != 0;
}

// The same with at most `polls` non-blocking tests: the fault-injection
// stand-in for a wait that runs out (test_wait returns at once, so a block
// that has just issued its copies gives up before they can have landed).
__device__ __forceinline__ bool test_phase0(uint32_t b, uint32_t polls)
{
    uint32_t ok = 0;
    for (uint32_t it = 0; it < polls && !ok; ++it)
        asm volatile("{\n .reg .pred P;\n mbarrier.test_wait.parity.shared::cta.b64 P, [%1], 0;\n selp.u32 %0, 1, 0, P;\n}"
                     : "=r"(ok) : "r"(b) : "memory");
    return ok != 0;
}

template <int NB, int kMinBlocks>
__global__ void __launch_bounds__(256, kMinBlocks) k_reduce_apply_staged(const StepArgs a, int64_t ahead)
{
    extern __shared__ __align__(128) uint8_t rows[];  // W rows of kRow bytes
    __shared__ __align__(8) uint64_t bar;
    constexpr int kGroupElems = 256 * kVec;          // elements per group (one per thread)
    constexpr int kRow = kStagedGroups * 256 * NB;   // wire bytes of one worker for the block
    const int64_t blk0 = static_cast<int64_t>(blockIdx.x) * (kStagedGroups * kGroupElems);
    if (threadIdx.x == 0) {
        const int64_t rem = a.d - blk0;
        const int64_t elems = rem < kStagedGroups * kGroupElems ? rem : kStagedGroups * kGroupElems;
        uint32_t bytes = static_cast<uint32_t>(((elems * NB + 7) / 8 + 15) / 16 * 16);
        // each worker's copy stays inside its padded row and the shared row
        if (!in_bounds(a, elems > 0 && bytes <= static_cast<uint32_t>(kRow) &&
                              blk0 * NB / 8 + bytes <= a.wire_stride * 4))
            bytes = 0;
        const uint32_t b = smem_addr(&bar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes * a.W) : "memory");
        const uint8_t* src = reinterpret_cast<const uint8_t*>(a.wire) + blk0 * NB / 8;
        const int64_t stride = a.wire_stride * 4;
        for (int i = 0; bytes > 0 && i < a.W; ++i)
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(smem_addr(rows + i * kRow)), "l"(src + i * stride), "r"(bytes), "r"(b)
                         : "memory");
    }
    // L2 is asked for the theta of the block `ahead` blocks later (about one
    // resident wave: the block that takes this slot next): measured 1.0-1.5 %
    // faster with signs from 16 workers and with 2-bit codes, neutral with
    // signs from 8; with 4-bit codes it was 2 % slower, so wider codes skip it
    if constexpr (NB <= 2) {
        const int64_t pblk = (static_cast<int64_t>(blockIdx.x) + ahead) * (kStagedGroups * kGroupElems);
#pragma unroll
        for (int q = 0; q < kStagedGroups; ++q) {
            const int64_t pe = pblk + q * kGroupElems + static_cast<int64_t>(threadIdx.x) * kVec;
            if (pe + kVec <= a.d)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.theta + pe));
        }
    }
    // every group's theta is requested while the wire bytes are in flight
    float th[kStagedGroups][kVec];
    int valid[kStagedGroups];
#pragma unroll
    for (int q = 0; q < kStagedGroups; ++q) {
        const int64_t e0 = blk0 + q * kGroupElems + static_cast<int64_t>(threadIdx.x) * kVec;
        valid[q] = e0 >= a.d ? 0 : ((a.d - e0 >= kVec) ? kVec : static_cast<int>(a.d - e0));
        if (valid[q] > 0)
            load_f32(a.theta, e0, valid[q], th[q]);
    }
    __shared__ float avg_tab[kAvgTab];
    fill_avg_table(a, avg_tab);
    __syncthreads();  // the barrier is initialised (and the table filled) before anyone polls it
    const uint32_t b = smem_addr(&bar);
    if (!(a.first_wait_polls ? test_phase0(b, a.first_wait_polls) : wait_phase0(b))) {
        if (threadIdx.x == 0)
            atomicOr(a.status, kStatusWaitTimeout);
        wait_phase0(b);  // drain this block's copies (full bounded wait) before leaving
        return;
    }
    using T = typename WireChunk<NB>::T;
#pragma unroll
    for (int q = 0; q < kStagedGroups; ++q) {
        if (valid[q] == 0)
            continue;
        int agg[kVec];
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            agg[j] = 0;
        uint32_t lo = 0, hi = 0;
        for (int i = 0; i < a.W; ++i)
            accumulate<NB>(agg, lo, hi, reinterpret_cast<const T*>(rows + i * kRow)[q * 256 + threadIdx.x]);
        if constexpr (NB == 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                agg[j] = 2 * static_cast<int>((lo >> (8 * j)) & 0xffu) - a.W;
                agg[j + 4] = 2 * static_cast<int>((hi >> (8 * j)) & 0xffu) - a.W;
            }
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            th[q][j] = lion_apply(th[q][j], direction(a, agg[j], avg_tab), a.lr, a.wd);
        store_f32(a.theta, blk0 + q * kGroupElems + static_cast<int64_t>(threadIdx.x) * kVec, valid[q], th[q]);
    }
}

template <int NB>
__global__ void __launch_bounds__(256) k_export_agg(const StepArgs a, int32_t* out)
{
    const int64_t e0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kVec;
    if (e0 >= a.d)
        return;
    const int valid = (a.d - e0 >= kVec) ? kVec : static_cast<int>(a.d - e0);
    if (!in_bounds(a, (e0 * NB) / 32 + (kVec * NB + 31) / 32 <= a.wire_stride))
        return;
    int agg[kVec];
    aggregate8<NB>(a, e0, agg);
    for (int j = 0; j < valid; ++j)
        out[e0 + j] = agg[j];
}

unsigned groups_grid(int64_t d)
{
    const int64_t groups = (d + kVec - 1) / kVec;
    return static_cast<unsigned>((groups + 255) / 256);
}

// Shared memory of the staged variant: W rows of kStagedGroups*256*NB bytes.  Above
// kStagedMaxBytes the register variant runs instead.
constexpr int kStagedMaxBytes = 64 * 1024;

// Blocks of the staged reduce that the whole device holds at once (6 per SM
// at its usual 40 registers), the distance of its theta prefetch.
int64_t prefetch_distance()
{
    static int64_t n = 0;
    if (n == 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
            n = static_cast<int64_t>(sms) * 6;
        else
            n = 152 * 6;
    }
    return n;
}

template <int NB, int kMinBlocks>
cudaError_t launch_staged(const StepArgs& a, int smem, cudaStream_t s)
{
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(k_reduce_apply_staged<NB, kMinBlocks>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
    }
    const int64_t per_block = static_cast<int64_t>(kStagedGroups) * 256 * kVec;
    const unsigned sgrid = static_cast<unsigned>((a.d + per_block - 1) / per_block);
    k_reduce_apply_staged<NB, kMinBlocks><<<sgrid, 256, smem, s>>>(a, prefetch_distance());
    return cudaGetLastError();
}

template <int NB>
cudaError_t launch_nb(const StepArgs& a, unsigned grid, cudaStream_t s)
{
    const int smem = a.W * kStagedGroups * 256 * NB;
    if (a.status != nullptr && smem <= kStagedMaxBytes) {
        // Signs from more than 8 workers: capping the kernel at 32 registers
        // (8 blocks per SM instead of 6) keeps more blocks waiting on their
        // copies at once; measured 4.5 % faster at W = 16 (GPT-2 medium) and
        // 0.2-0.7 % slower at W = 8, so only the larger vote takes it.
        if constexpr (NB == 1) {
            if (a.W > 8)
                return launch_staged<NB, 8>(a, smem, s);
        }
        return launch_staged<NB, 1>(a, smem, s);
    } else {
        k_reduce_apply<NB><<<grid, 256, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reduce_apply(const StepArgs& a, int l1_mode, cudaStream_t s)
{
    if (a.d == 0)
        return cudaSuccess;
    const unsigned grid = groups_grid(a.d);
    switch (l1_mode ? a.nbits : 1) {
    case 1: return launch_nb<1>(a, grid, s);
    case 2: return launch_nb<2>(a, grid, s);
    case 4: return launch_nb<4>(a, grid, s);
    case 8: return launch_nb<8>(a, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_export_agg(const StepArgs& a, int l1_mode, int32_t* agg, cudaStream_t s)
{
    if (a.d == 0)
        return cudaSuccess;
    const unsigned grid = groups_grid(a.d);
    switch (l1_mode ? a.nbits : 1) {
    case 1: k_export_agg<1><<<grid, 256, 0, s>>>(a, agg); break;
    case 2: k_export_agg<2><<<grid, 256, 0, s>>>(a, agg); break;
    case 4: k_export_agg<4><<<grid, 256, 0, s>>>(a, agg); break;
    case 8: k_export_agg<8><<<grid, 256, 0, s>>>(a, agg); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace lc
