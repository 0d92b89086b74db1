// compress.cu -- per-worker compression pass of the compressed Lion step.
//
// 8 consecutive elements per thread.  For one worker the thread loads 8
// gradients and 8 momenta, forms the update vector c ("Lion Cub: Minimizing
// Communication Overhead in Distributed Lion", "What carries the argument"),
// emits the wire bits -- a 0/1 sign with exact zeros sent as the step's
// alternating sign, or the Eq. (1) L1 code -- and writes the worker's new
// momentum.  Unsynchronized tiles run one block per (tile, worker).  On
// tensors whose momentum is synchronized this step a block takes all
// workers of its tile in order, sums their new momenta in registers and
// writes the mean to every worker, so the sync costs no extra memory pass.
//
// Wire packing (LSB first): a thread's 8 elements hold 8*NB bits.  For the
// 1-bit sign, four neighbouring lanes' bytes form one 32-bit word; for 2-bit
// codes two lanes' halves; 4-bit codes fill one word per thread; 8-bit codes
// two words.
#include "compress_common.cuh"

namespace lc {
namespace {

// Tiles whose momentum is not synchronized this step: one block per (tile,
// worker) -- grid (tiles, W) -- so each thread handles one worker's 8
// elements with no loop, which keeps registers low: 8 blocks of 256 threads
// per SM (at most 32 registers), the full 2048 threads.
//
// With L1 codes each block first asks L2 for the tile `ahead` blocks later of
// the same worker -- one resident wave of blocks ahead, the block that will
// take this slot next -- so that block's loads find its lines on the way:
// measured 0.35 % faster on the 2-bit 1.3B workload and 0.14 % on the 4-bit
// GPT-2-medium one; with 1-bit signs it was 0.2-0.3 % slower, so signs skip
// it, and 8-bit codes do too (there it would spill under the 32-register cap).
template <typename GT, int NB>
__global__ void __launch_bounds__(kThreads, 8) k_compress(const StepArgs a, int64_t tile0, int64_t ahead)
{
    const int64_t tix = tile0 + blockIdx.x;
    const Tile tl = in_bounds(a, tix < a.ntiles) ? a.tiles[tix] : Tile{0, 0, 0u};
    const int i = blockIdx.y;
    if constexpr (NB == 2 || NB == 4) {
        const int64_t pix = tix + ahead;
        if (pix < tile0 + gridDim.x && in_bounds(a, pix < a.ntiles)) {
            const Tile pt = a.tiles[pix];
            const int64_t pe = pt.start + static_cast<int64_t>(threadIdx.x) * kVec;
            if (pe + kVec <= pt.start + pt.len) {
                asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const GT*>(a.g[i]) + pe));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.m[i] + pe));
            }
        }
    }
    const int64_t e0 = tl.start + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = tl.start + tl.len - e0;
    const int valid = checked_valid<NB>(a, e0, left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left)));
    float g[kVec], m[kVec];
    if (valid > 0) {
        load_gm<GT>(a.g[i], a.m[i], e0, valid, g, m);
    } else {
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            g[j] = m[j] = 0.0f;
    }
    float inv = 0.0f;
    if constexpr (NB > 1) {
        const uint32_t k = tl.meta & ~kTileSync;
        if (in_bounds(a, k < static_cast<uint32_t>(a.K)))
            inv = a.inv[static_cast<int64_t>(i) * a.K + k];
    }
    const uint64_t bits = compress8<NB>(a, g, m, valid, inv);
    store_wire<NB>(a.wire + static_cast<int64_t>(i) * a.wire_stride, e0, valid, bits);
    if (valid > 0)
        store_f32(a.m[i], e0, valid, m);
}

// Tiles of synchronized tensors on a sync step: one block per tile, the
// thread loops over the workers in order, summing their new momenta in
// registers, and writes the mean to every worker (no extra memory pass).
// Each iteration asks L2 for the gradients and momenta of the worker two
// ahead (prefetch instructions hold no registers), so the loop's loads
// mostly hit L2 while DRAM streams the next ones; at 40 registers six blocks
// fit an SM.  Measured on the 16-worker GPT-2-medium workload against
// keeping the next worker's loads in registers (63 registers, four blocks):
// the sync tiles' pass ran about 5 % faster, at the plain tiles' rate.
template <typename GT, int NB>
__global__ void __launch_bounds__(kThreads, 6) k_compress_sync(const StepArgs a, int64_t tile0)
{
    constexpr int kAhead = 2;
    const int64_t tix = tile0 + blockIdx.x;
    const Tile tl = in_bounds(a, tix < a.ntiles) ? a.tiles[tix] : Tile{0, 0, 0u};
    const int64_t e0 = tl.start + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = tl.start + tl.len - e0;
    const int valid = checked_valid<NB>(a, e0, left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left)));
    int k = static_cast<int>(tl.meta & ~kTileSync);
    if (!in_bounds(a, k < a.K))
        k = 0;

    float acc[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j)
        acc[j] = 0.0f;
    if (valid == kVec) {
#pragma unroll
        for (int q = 0; q < kAhead; ++q) {
            if (q < a.W) {
                asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const GT*>(a.g[q]) + e0));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.m[q] + e0));
            }
        }
    }
    for (int i = 0; i < a.W; ++i) {
        if (valid == kVec && i + kAhead < a.W) {
            const int q = i + kAhead;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const GT*>(a.g[q]) + e0));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a.m[q] + e0));
        }
        float g[kVec], m[kVec];
        if (valid > 0) {
            load_gm<GT>(a.g[i], a.m[i], e0, valid, g, m);
        } else {
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                g[j] = m[j] = 0.0f;
        }
        float inv = 0.0f;
        if constexpr (NB > 1)
            inv = a.inv[static_cast<int64_t>(i) * a.K + k];
        const uint64_t bits = compress8<NB>(a, g, m, valid, inv);
        store_wire<NB>(a.wire + static_cast<int64_t>(i) * a.wire_stride, e0, valid, bits);
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            acc[j] = (i == 0) ? m[j] : __fadd_rn(acc[j], m[j]);
    }
    if (valid > 0) {
        const float fw = static_cast<float>(a.W);
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            acc[j] = __fdiv_rn(acc[j], fw);
        for (int i = 0; i < a.W; ++i)
            store_f32(a.m[i], e0, valid, acc);
    }
}

// Blocks of k_compress resident on the whole device at once (8 per SM).
int64_t resident_blocks()
{
    static int64_t n = 0;
    if (n == 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
            n = static_cast<int64_t>(sms) * 8;
        else
            n = 152 * 8;
    }
    return n;
}

template <typename GT, int NB>
cudaError_t launch_nb(const StepArgs& a, cudaStream_t s)
{
    // Tiles [0, nplain) belong to unsynchronized tensors, [nplain, ntiles)
    // to synchronized ones; off sync steps every tile takes the plain kernel.
    const int64_t nplain = a.sync_now ? a.nplain : a.ntiles;
    if (nplain > 0)
        k_compress<GT, NB><<<dim3(static_cast<unsigned>(nplain), a.W), kThreads, 0, s>>>(a, 0, resident_blocks());
    if (a.ntiles > nplain)
        k_compress_sync<GT, NB><<<static_cast<unsigned>(a.ntiles - nplain), kThreads, 0, s>>>(a, nplain);
    return cudaGetLastError();
}

template <typename GT>
cudaError_t launch_typed(const StepArgs& a, int nb, cudaStream_t s)
{
    switch (nb) {
    case 1: return launch_nb<GT, 1>(a, s);
    case 2: return launch_nb<GT, 2>(a, s);
    case 4: return launch_nb<GT, 4>(a, s);
    case 8: return launch_nb<GT, 8>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_compress(const StepArgs& a, int grad_dtype, int l1_mode, cudaStream_t s)
{
    if (a.ntiles == 0)
        return cudaSuccess;
    const int nb = l1_mode ? a.nbits : 1;
    if (grad_dtype == LIONCUB_GRAD_BF16)
        return launch_typed<__nv_bfloat16>(a, nb, s);
    return launch_typed<float>(a, nb, s);
}

}  // namespace lc
