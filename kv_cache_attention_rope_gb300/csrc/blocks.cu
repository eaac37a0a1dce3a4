// Copy-on-write of shared cache blocks.
//
// "Nano-vLLM Part 2" page, section 05: the block manager keeps reference
// counts so that sequences with a common prefix share its blocks, and one
// block id names the same block in every layer's K and V area.  When a
// sequence appends into a partially filled block that another sequence still
// references, the block is first duplicated under a fresh id; this kernel
// makes those duplicates, for every K and V region at once.
//
// Plain 16-byte vector copies, grid-stride over (pair, region, vector): each
// block-region is a contiguous Hkv x block_size x D run, so every warp reads
// and writes 512 contiguous bytes.  A pair with an id outside the pool is
// skipped and recorded as KVATTN_ERR_BAD_INDEX.
#include <algorithm>

#include "kvattn_internal.cuh"

namespace kvattn {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const __grid_constant__ CopyArgs a)
{
    pdl_wait();
    const int64_t vpb = a.block_bytes / 16;             // vectors per block-region
    const int64_t regions = 2 * (int64_t)a.layers;
    const int64_t total = (int64_t)a.n * regions * vpb;
    for (int64_t v = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x; v < total;
         v += (int64_t)gridDim.x * kCopyThreads) {
        const int64_t pair = v / (regions * vpb);
        const int64_t rem = v - pair * regions * vpb;
        const int64_t r = rem / vpb, off = rem - r * vpb;
        const int32_t s = a.src[pair], d = a.dst[pair];
        if (s < 0 || s >= a.num_blocks || d < 0 || d >= a.num_blocks) {
            if (r == 0 && off == 0) record_error(a.status, KVATTN_ERR_BAD_INDEX);
            continue;
        }
        char* base = ((r & 1) ? a.v_base : a.k_base) + (r >> 1) * a.layer_stride;
        const uint4 x = *reinterpret_cast<const uint4*>(base + (int64_t)s * a.block_bytes + off * 16);
        *reinterpret_cast<uint4*>(base + (int64_t)d * a.block_bytes + off * 16) = x;
    }
}

}  // namespace

kvattn_status launch_copy_blocks(const CopyArgs& a, cudaStream_t s)
{
    const int64_t total = (int64_t)a.n * 2 * a.layers * (a.block_bytes / 16);
    const int64_t want = (total + kCopyThreads - 1) / kCopyThreads;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms() * 8));
    const cudaError_t e0 = launch_pdl(copy_blocks_kernel, dim3(grid), dim3(kCopyThreads), 0, s, a);
    if (e0 != cudaSuccess) return cuda_status(e0);
    return cuda_status(cudaGetLastError());
}

}  // namespace kvattn
