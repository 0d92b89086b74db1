// dist.cu -- kernels of the data-parallel exchange: the compressed Lion step
// with the W workers spread over several ranks (one GPU each), every rank
// holding W/N of them and a copy of theta.
//
// "Lion Cub: Minimizing Communication Overhead in Distributed Lion": the
// quoted body text on the implementation (1-bit Lion Cub exchanges its packed
// signs with an AlltoAll, the 4-bit and wider variants sum their codes with
// an AllReduce), "What carries the argument" (an allreduce of 1-bit words
// built for the majority vote; the workers' quantized update vectors are
// summed and the sum's sign is applied; the embedding and output layers
// average their momentum) and the
// Fig. 1 / Fig. 8 captions (1-bit and p-bit containers).
//
// A step is three launches around the caller's collectives:
//   sign mode  compress (wire words chunk-major into the send buffer)
//              | all-to-all: rank r receives every worker's words of chunk r
//              owner reduce (vote of chunk r -> 2-bit directions, or the vote
//              sum for the average)
//              | allgather of the directions
//              apply (theta from the directions)
//   L1 mode    M1, compress (codes into the rank's own wire rows)
//              code sum of the rank's workers (int8 or int32 per element)
//              | allreduce (sum)
//              apply (theta from the sign of the sum)
// On sync steps the compress pass writes the new momenta of synchronized
// tensors to a sync buffer instead of the momenta; after the caller's
// allgather of those buffers the apply launch averages them in worker order
// (s = m_0; s += m_j for j = 1..W-1; m = s / W), exactly as one GPU does.
#include "aggregate.cuh"
#include "compress_common.cuh"

namespace lc {
namespace {

// The pass over one (tile, local worker): c, the wire field, the new
// momentum.  Wire words: chunk-major in sign mode (element e of local worker
// i goes to row (e / chunk) * W + i, bit (e % chunk) of that row, so the
// buffer's segment r is what rank r receives), one row per worker in L1
// mode.  Momenta of synchronized tiles go to the sync buffer on sync steps.
template <typename GT, int NB>
__global__ void __launch_bounds__(kThreads, 8) k_compress_dist(const StepArgs a)
{
    const int64_t tix = blockIdx.x;
    const Tile tl = in_bounds(a, tix < a.ntiles) ? a.tiles[tix] : Tile{0, 0, 0u};
    const int i = blockIdx.y;
    const int64_t e0 = tl.start + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = tl.start + tl.len - e0;
    int valid = left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left));
    if (valid > 0 && !in_bounds(a, e0 >= 0 && e0 + valid <= a.d))
        valid = 0;

    // wire row and the element's position in it (sign mode is chunk-major,
    // L1 mode has one row per worker)
    uint32_t* row;
    int64_t er;
    if constexpr (NB == 1) {
        // chunk is a multiple of 4096 and a 32-element word never spans two chunks
        const int64_t c = static_cast<int64_t>(static_cast<uint32_t>(e0 >> 12) /
                                               static_cast<uint32_t>(a.chunk >> 12));
        row = a.wire + (c * a.W + i) * a.chunk_words;
        er = e0 - c * a.chunk;
        if (valid > 0 && !in_bounds(a, (er * NB) / 32 < a.chunk_words))
            valid = 0;
    } else {
        row = a.wire + static_cast<int64_t>(i) * a.wire_stride;
        er = e0;
        if (valid > 0 && !in_bounds(a, (er * NB) / 32 + (kVec * NB + 31) / 32 <= a.wire_stride))
            valid = 0;
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
    if constexpr (NB > 1) {
        const uint32_t k = tl.meta & ~kTileSync;
        if (in_bounds(a, k < static_cast<uint32_t>(a.K)))
            inv = a.inv[static_cast<int64_t>(i) * a.K + k];
    }
    const uint64_t bits = compress8<NB>(a, g, m, valid, inv);
    store_wire<NB>(row, er, valid, bits);
    if (valid > 0) {
        if (a.sync_now && (tl.meta & kTileSync)) {
            const int64_t slot = (tix - a.nplain) * kTile + static_cast<int64_t>(threadIdx.x) * kVec;
            if (in_bounds(a, tix >= a.nplain && slot + valid <= a.sync_slots))
                store_f32(a.sync_buf + static_cast<int64_t>(i) * a.sync_slots, slot, valid, m);
        } else {
            store_f32(a.m[i], e0, valid, m);
        }
    }
}

// The chunk owner's vote: a.wire holds the W received rows of chunk_words
// words (a.wire_stride), a.d the chunk's length.  Per element the direction
// of the global sign (DB = 2: two's-complement -1, 0, +1, ties taking tie_u)
// or the vote sum itself (DB = 8, for the average, |sum| <= W <= 127).
template <int DB>
__global__ void __launch_bounds__(256) k_owner_reduce(const StepArgs a, void* dir)
{
    const int64_t e0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kVec;
    if (e0 >= a.d)
        return;
    const int valid = (a.d - e0 >= kVec) ? kVec : static_cast<int>(a.d - e0);
    if (!in_bounds(a, e0 / 32 < a.wire_stride))
        return;
    int agg[kVec];
    aggregate8<1>(a, e0, agg);
    const int tie = static_cast<int>(a.tie_u);
    if constexpr (DB == 2) {
        uint32_t f = 0;
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int s = agg[j] > 0 ? 1 : (agg[j] < 0 ? -1 : tie);
            if (j < valid)
                f |= (static_cast<uint32_t>(s) & 3u) << (2 * j);
        }
        static_cast<uint16_t*>(dir)[e0 >> 3] = static_cast<uint16_t>(f);
    } else {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            lo |= (static_cast<uint32_t>(agg[j]) & 0xffu) << (8 * j);
            hi |= (static_cast<uint32_t>(agg[j + 4]) & 0xffu) << (8 * j);
        }
        reinterpret_cast<uint2*>(static_cast<uint8_t*>(dir) + e0)[0] = make_uint2(lo, hi);
    }
}

// The L1 codes of the rank's own workers summed per element (int8 when the
// full sum fits, W * qmax <= 127, else int32), ready for the allreduce.
template <int NB, typename AT>
__global__ void __launch_bounds__(256) k_code_sum_local(const StepArgs a, AT* agg_out)
{
    const int64_t e0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kVec;
    if (e0 >= a.d)
        return;
    const int valid = (a.d - e0 >= kVec) ? kVec : static_cast<int>(a.d - e0);
    if (!in_bounds(a, (e0 * NB) / 32 + (kVec * NB + 31) / 32 <= a.wire_stride))
        return;
    int agg[kVec];
    aggregate8<NB>(a, e0, agg);
    if (valid == kVec) {
        if constexpr (sizeof(AT) == 1) {
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo |= (static_cast<uint32_t>(agg[j]) & 0xffu) << (8 * j);
                hi |= (static_cast<uint32_t>(agg[j + 4]) & 0xffu) << (8 * j);
            }
            reinterpret_cast<uint2*>(agg_out + e0)[0] = make_uint2(lo, hi);
        } else {
            int4* p = reinterpret_cast<int4*>(agg_out + e0);
            p[0] = make_int4(agg[0], agg[1], agg[2], agg[3]);
            p[1] = make_int4(agg[4], agg[5], agg[6], agg[7]);
        }
    } else {
        for (int j = 0; j < valid; ++j)
            agg_out[e0 + j] = static_cast<AT>(agg[j]);
    }
}

// theta from the gathered directions (DB = 2) or vote sums (DB = 8, the
// D-Lion average u = RN(sum / W) from the block's table of quotients).
template <int DB>
__global__ void __launch_bounds__(256) k_apply_dir(const StepArgs a, const void* dir)
{
    __shared__ float avg_tab[kAvgTab];
    fill_avg_table(a, avg_tab);
    __syncthreads();
    const int64_t e0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kVec;
    if (e0 >= a.d)
        return;
    const int valid = (a.d - e0 >= kVec) ? kVec : static_cast<int>(a.d - e0);
    float th[kVec];
    load_f32(a.theta, e0, valid, th);
    float u[kVec];
    if constexpr (DB == 2) {
        const uint32_t f = static_cast<const uint16_t*>(dir)[e0 >> 3];
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            u[j] = static_cast<float>(static_cast<int32_t>(f << (30 - 2 * j)) >> 30);
    } else {
        const uint2 v = reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(dir) + e0)[0];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            u[j] = direction(a, static_cast<int32_t>(v.x << (24 - 8 * j)) >> 24, avg_tab);
            u[j + 4] = direction(a, static_cast<int32_t>(v.y << (24 - 8 * j)) >> 24, avg_tab);
        }
    }
#pragma unroll
    for (int j = 0; j < kVec; ++j)
        th[j] = lion_apply(th[j], u[j], a.lr, a.wd);
    store_f32(a.theta, e0, valid, th);
}

// theta from the all-reduced code sums: the global sign, ties taking tie_u.
template <typename AT>
__global__ void __launch_bounds__(256) k_apply_agg(const StepArgs a, const AT* agg)
{
    const int64_t e0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kVec;
    if (e0 >= a.d)
        return;
    const int valid = (a.d - e0 >= kVec) ? kVec : static_cast<int>(a.d - e0);
    float th[kVec];
    load_f32(a.theta, e0, valid, th);
    int v[kVec];
    if (valid == kVec) {
        if constexpr (sizeof(AT) == 1) {
            const uint2 w = reinterpret_cast<const uint2*>(agg + e0)[0];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[j] = static_cast<int32_t>(w.x << (24 - 8 * j)) >> 24;
                v[j + 4] = static_cast<int32_t>(w.y << (24 - 8 * j)) >> 24;
            }
        } else {
            const int4* p = reinterpret_cast<const int4*>(agg + e0);
            const int4 x = p[0], y = p[1];
            v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            v[j] = j < valid ? static_cast<int>(agg[e0 + j]) : 0;
    }
#pragma unroll
    for (int j = 0; j < kVec; ++j)
        th[j] = lion_apply(th[j], direction(a, v[j], nullptr), a.lr, a.wd);
    store_f32(a.theta, e0, valid, th);
}

// Momentum sync after the allgather: recv holds W_global rows of sync_slots
// new momenta (worker order); each synchronized element's mean goes to every
// local worker's momentum.  One block per synchronized tile.
__global__ void __launch_bounds__(kThreads) k_sync_mean(const StepArgs a, int W_global, const float* recv)
{
    const int64_t tix = a.nplain + blockIdx.x;
    const Tile tl = in_bounds(a, tix < a.ntiles) ? a.tiles[tix] : Tile{0, 0, 0u};
    const int64_t e0 = tl.start + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = tl.start + tl.len - e0;
    int valid = left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left));
    const int64_t slot = static_cast<int64_t>(blockIdx.x) * kTile + static_cast<int64_t>(threadIdx.x) * kVec;
    if (valid > 0 && !in_bounds(a, e0 + valid <= a.d && slot + valid <= a.sync_slots))
        valid = 0;
    if (valid == 0)
        return;
    float s[kVec];
    for (int j = 0; j < W_global; ++j) {
        float v[kVec];
        load_f32(recv + static_cast<int64_t>(j) * a.sync_slots, slot, valid, v);
#pragma unroll
        for (int q = 0; q < kVec; ++q)
            s[q] = (j == 0) ? v[q] : __fadd_rn(s[q], v[q]);
    }
    const float fw = static_cast<float>(W_global);
#pragma unroll
    for (int q = 0; q < kVec; ++q)
        s[q] = __fdiv_rn(s[q], fw);
    for (int i = 0; i < a.W; ++i)
        store_f32(a.m[i], e0, valid, s);
}

unsigned groups_grid(int64_t n)
{
    const int64_t groups = (n + kVec - 1) / kVec;
    return static_cast<unsigned>((groups + 255) / 256);
}

template <typename GT>
cudaError_t compress_typed(const StepArgs& a, int nb, cudaStream_t s)
{
    const dim3 grid(static_cast<unsigned>(a.ntiles), a.W);
    switch (nb) {
    case 1: k_compress_dist<GT, 1><<<grid, kThreads, 0, s>>>(a); break;
    case 2: k_compress_dist<GT, 2><<<grid, kThreads, 0, s>>>(a); break;
    case 4: k_compress_dist<GT, 4><<<grid, kThreads, 0, s>>>(a); break;
    case 8: k_compress_dist<GT, 8><<<grid, kThreads, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int NB>
cudaError_t code_sum_nb(const StepArgs& a, int agg_bytes, void* agg, unsigned grid, cudaStream_t s)
{
    if (agg_bytes == 1)
        k_code_sum_local<NB, int8_t><<<grid, 256, 0, s>>>(a, static_cast<int8_t*>(agg));
    else
        k_code_sum_local<NB, int32_t><<<grid, 256, 0, s>>>(a, static_cast<int32_t*>(agg));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compress_dist(const StepArgs& a, int grad_dtype, int l1_mode, cudaStream_t s)
{
    if (a.ntiles == 0)
        return cudaSuccess;
    const int nb = l1_mode ? a.nbits : 1;
    if (grad_dtype == LIONCUB_GRAD_BF16)
        return compress_typed<__nv_bfloat16>(a, nb, s);
    return compress_typed<float>(a, nb, s);
}

cudaError_t launch_owner_reduce(const StepArgs& a, int dir_bits, void* dir, cudaStream_t s)
{
    if (a.d <= 0)
        return cudaSuccess;
    if (dir_bits == 2)
        k_owner_reduce<2><<<groups_grid(a.d), 256, 0, s>>>(a, dir);
    else if (dir_bits == 8)
        k_owner_reduce<8><<<groups_grid(a.d), 256, 0, s>>>(a, dir);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_code_sum_local(const StepArgs& a, int agg_bytes, void* agg, cudaStream_t s)
{
    if (a.d <= 0)
        return cudaSuccess;
    if (agg_bytes != 1 && agg_bytes != 4)
        return cudaErrorInvalidValue;
    const unsigned grid = groups_grid(a.d);
    switch (a.nbits) {
    case 2: return code_sum_nb<2>(a, agg_bytes, agg, grid, s);
    case 4: return code_sum_nb<4>(a, agg_bytes, agg, grid, s);
    case 8: return code_sum_nb<8>(a, agg_bytes, agg, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_apply_dir(const StepArgs& a, int dir_bits, const void* dir, cudaStream_t s)
{
    if (a.d <= 0)
        return cudaSuccess;
    if (dir_bits == 2)
        k_apply_dir<2><<<groups_grid(a.d), 256, 0, s>>>(a, dir);
    else if (dir_bits == 8)
        k_apply_dir<8><<<groups_grid(a.d), 256, 0, s>>>(a, dir);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_apply_agg(const StepArgs& a, int agg_bytes, const void* agg, cudaStream_t s)
{
    if (a.d <= 0)
        return cudaSuccess;
    if (agg_bytes == 1)
        k_apply_agg<int8_t><<<groups_grid(a.d), 256, 0, s>>>(a, static_cast<const int8_t*>(agg));
    else if (agg_bytes == 4)
        k_apply_agg<int32_t><<<groups_grid(a.d), 256, 0, s>>>(a, static_cast<const int32_t*>(agg));
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_sync_mean(const StepArgs& a, int W_global, const float* recv, cudaStream_t s)
{
    const int64_t nsync = a.ntiles - a.nplain;
    if (nsync <= 0)
        return cudaSuccess;
    k_sync_mean<<<static_cast<unsigned>(nsync), kThreads, 0, s>>>(a, W_global, recv);
    return cudaGetLastError();
}

}  // namespace lc
