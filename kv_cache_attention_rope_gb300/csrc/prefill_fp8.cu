// Chunked prefill over the fp8 (e4m3) page cache.
//
// What it computes: the causal chunk attention of kvattn_prefill_chunk
// ("From-scratch AI inference engine" page, sections 3.3 and 3.4) with K and
// V the dequantised cache values code * scale ("Tokenizer, KV Cache and
// RoPE" page, section 2: the cache holds values compressed to 8 bits).
//
// How (GB300 design): chunked prefill is bound by the tensor cores, not by
// HBM (a 16-chunk step of 512 queries over 4K-token prefixes does ~6e11
// FLOPs against ~0.3 GB of bf16 K/V), so the fp8 pages of the chunks'
// blocks are first expanded into a bf16 copy in the caller's workspace and
// the bf16 tcgen05 prefill kernel runs over that copy unchanged.  Converting
// inside the prefill kernel would put ~3 instructions per K/V element on the
// SMs whose softmax warps already bound that kernel, and its shared memory
// has no room for a raw-page stage; the copy costs one pass over the fp8
// pages and the bf16 writes, at HBM speed.
//  - prefill_fp8_plan (one CTA): blocks each chunk's keys occupy,
//    ceil((prefix + chunk length) / block_size); their exclusive prefix sum
//    (the chunk's first block in the copy); the owning chunk of every copy
//    block; and the copy's block table (chunk c, column j -> first[c] + j).
//  - prefill_fp8_expand (persistent warps): one warp per 16-token page of
//    one KV head.  Each warp takes a contiguous range of copy pages; its
//    lanes look up 32 pages' sources at once, then the warp streams the pages
//    through two shared-memory buffers (16-byte asynchronous copies of page
//    i + 1 fly while page i converts) and converts them: K rows un-swizzled,
//    V transposed back to token-major
//    rows, every element written as bf16(code * scale) (the product in fp32,
//    RN, then RN to bf16).  Only pages holding keys the prefill reads are
//    converted; the prefill zeroes stale V rows of a sequence's last page
//    itself.
#include <algorithm>
#include <cstring>

#include <cuda_fp16.h>

#include "kvattn_tc.cuh"

namespace kvattn {
namespace {

constexpr int kF8D = 128;  // head dim of the fp8 page layout

struct Fp8PrefillArgs {
    const unsigned char* pool;
    int64_t num_blocks;        // of the fp8 cache
    const int32_t* block_table;
    const int32_t* cu_q_lens;
    const int32_t* prefix_lens;
    int32_t num_chunks, max_blocks, max_q_len, total_q, block_size, hkv;
    int64_t nb;                // blocks of the bf16 copy
    int64_t* first;            // [num_chunks + 1]
    int32_t* owner;            // [nb]
    int32_t* ctable;           // [num_chunks][max_blocks]
    __nv_bfloat16* k_copy;     // [nb][hkv][block_size][128]
    __nv_bfloat16* v_copy;
    int* status;
};

// Blocks chunk c's keys occupy; 0 for a chunk the prefill kernel rejects or
// skips (it records the error itself).
__device__ __forceinline__ int chunk_blocks(const Fp8PrefillArgs& a, int c)
{
    const int q0 = a.cu_q_lens[c], qlen = a.cu_q_lens[c + 1] - q0, P = a.prefix_lens[c];
    if (qlen <= 0 || P < 0 || qlen > a.max_q_len || q0 < 0 || q0 + qlen > a.total_q ||
        (int64_t)P + qlen > (int64_t)a.max_blocks * a.block_size)
        return 0;
    return (P + qlen + a.block_size - 1) / a.block_size;
}

__global__ void __launch_bounds__(1024) prefill_fp8_plan(const Fp8PrefillArgs a)
{
    pdl_wait();
    __shared__ int64_t wsum[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int64_t carry = 0;
    for (int base = 0; base < a.num_chunks; base += 1024) {
        const int c = base + tid;
        const int64_t n = c < a.num_chunks ? chunk_blocks(a, c) : 0;
        int64_t x = n;  // inclusive scan over the warp, then over the warps
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int64_t w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        if (c < a.num_chunks) a.first[c] = carry + x - n + (warp > 0 ? wsum[warp - 1] : 0);
        carry += wsum[31];
        __syncthreads();  // wsum is rewritten by the next round
    }
    if (tid == 0) a.first[a.num_chunks] = carry;
    __syncthreads();
    // owners and the copy's block table: one warp per chunk, lanes over its blocks
    for (int c = warp; c < a.num_chunks; c += 32) {
        const int64_t f = a.first[c];
        const int n = (int)(a.first[c + 1] - f);
        int32_t* trow = a.ctable + (int64_t)c * a.max_blocks;
        for (int j = lane; j < n; j += 32) {
            const int64_t b = f + j;
            if (b < a.nb) {
                a.owner[b] = c;
                trow[j] = (int32_t)b;
            } else {
                trow[j] = -1;  // more key blocks than the copy was sized for
                record_error(a.status, KVATTN_ERR_BAD_INDEX);
            }
        }
    }
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h)
{
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi)
{
    const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&r);
}

// Four e4m3 codes (bytes of w) times s -> two bf16 pairs
__device__ __forceinline__ void expand4(uint32_t w, float s, uint32_t& o0, uint32_t& o1)
{
    const float2 a = f16x2_to_float2(e4m3x2_to_f16x2(w));
    const float2 b = f16x2_to_float2(e4m3x2_to_f16x2(w >> 16));
    o0 = bf16x2_rn(a.x * s, a.y * s);
    o1 = bf16x2_rn(b.x * s, b.y * s);
}

constexpr int kExpandWarps = 8;

__global__ void __launch_bounds__(kExpandWarps * 32) prefill_fp8_expand(const Fp8PrefillArgs a)
{
    pdl_wait();
    extern __shared__ __align__(16) unsigned char bufs[];  // [kExpandWarps][2][kF8Page]
    const int lane = threadIdx.x & 31;
    unsigned char* pbuf = bufs + (threadIdx.x >> 5) * 2 * kF8Page;
    const int ppb = a.block_size / 16;  // pages per block and head
    const int64_t used = min(a.first[a.num_chunks], a.nb);
    const int64_t pages = used * a.hkv * ppb;
    const int64_t nwarps = (int64_t)gridDim.x * kExpandWarps;
    const int64_t wid = (int64_t)blockIdx.x * kExpandWarps + (threadIdx.x >> 5);
    const int64_t per = (pages + nwarps - 1) / nwarps;
    const int64_t beg = wid * per, end = min(pages, beg + per);
    for (int64_t g0 = beg; g0 < end; g0 += 32) {
        // lane i: source page of copy page g0 + i (null when it is not needed)
        const unsigned char* my_src = nullptr;
        const int64_t g = g0 + lane;
        if (g < end) {
            const int64_t b = g / (a.hkv * ppb);
            const int rem = (int)(g - b * a.hkv * ppb), h = rem / ppb, p = rem - h * ppb;
            const int c = a.owner[b];
            const int j = (int)(b - a.first[c]);
            const int total = a.prefix_lens[c] + a.cu_q_lens[c + 1] - a.cu_q_lens[c];
            if (j * a.block_size + p * 16 < total) {
                const int32_t blk = a.block_table[(int64_t)c * a.max_blocks + j];
                if (blk < 0 || blk >= a.num_blocks)
                    record_error(a.status, KVATTN_ERR_BAD_INDEX);
                else
                    my_src = a.pool + (((int64_t)blk * a.hkv + h) * ppb + p) * kF8Page;
            }
        }
        // pages to convert: the set bits of `todo` (lane i: copy page g0 + i);
        // each is copied whole into this warp's shared buffer with 16-byte
        // asynchronous copies, the next one while the current one converts
        unsigned todo = __ballot_sync(0xffffffffu, my_src != nullptr);
        auto fetch = [&](int i, int bsel) {
            const unsigned char* src = reinterpret_cast<const unsigned char*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(my_src), i));
            const uint32_t dst = smem_addr(pbuf + bsel * kF8Page);
            for (int c = lane; c < kF8Page / 16; c += 32)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16 * c), "l"(src + 16 * c)
                             : "memory");
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        int bsel = 0;
        if (todo) fetch(__ffs(todo) - 1, 0);
        while (todo) {
            const int i = __ffs(todo) - 1;
            todo &= todo - 1;
            if (todo) {
                fetch(__ffs(todo) - 1, bsel ^ 1);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
            __syncwarp();  // every lane's copies of page i have landed
            const unsigned char* src = pbuf + bsel * kF8Page;
            // copy page g0 + i = rows 16 p .. 16 p + 15 of copy block b, head h:
            // [b][h][block_size][128] has them at ((b * hkv + h) * ppb + p) * 16 rows
            const int64_t row0 = (g0 + i) * 16;
            __nv_bfloat16* kd = a.k_copy + row0 * kF8D;
            __nv_bfloat16* vd = a.v_copy + row0 * kF8D;
            const float* scales = reinterpret_cast<const float*>(src + kF8KsOff);
            // K: lane takes chunk cc (16 dims) of tokens r = lane / 8 + 4 t
            const int cc = lane & 7;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int r = (lane >> 3) + 4 * t;
                const uint4 kw = *reinterpret_cast<const uint4*>(src + r * 128 + 16 * (cc ^ f8_swz(r)));
                const float ks = scales[r];
                uint4 o0, o1;
                expand4(kw.x, ks, o0.x, o0.y);
                expand4(kw.y, ks, o0.z, o0.w);
                expand4(kw.z, ks, o1.x, o1.y);
                expand4(kw.w, ks, o1.z, o1.w);
                *reinterpret_cast<uint4*>(kd + r * kF8D + 16 * cc) = o0;
                *reinterpret_cast<uint4*>(kd + r * kF8D + 16 * cc + 8) = o1;
            }
            // V: lane takes dims 8 gv .. 8 gv + 7 of tokens 8 hv .. 8 hv + 7
            const int gv = lane >> 1, hv = lane & 1;
            uint2 vw[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                vw[k] = *reinterpret_cast<const uint2*>(src + kF8VOff + 16 * (8 * gv + k) + 8 * hv);
            const float4 vs0 = *reinterpret_cast<const float4*>(src + kF8VsOff + 32 * hv);
            const float4 vs1 = *reinterpret_cast<const float4*>(src + kF8VsOff + 32 * hv + 16);
            const float vs[8] = {vs0.x, vs0.y, vs0.z, vs0.w, vs1.x, vs1.y, vs1.z, vs1.w};
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) {
                // token 8 hv + tt: byte tt % 4 of the low (tt < 4) or high word of each dim
                const uint32_t sel = (uint32_t)(tt & 3) | ((uint32_t)(4 + (tt & 3)) << 4);
                uint32_t o[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t x = tt < 4 ? vw[2 * m].x : vw[2 * m].y;
                    const uint32_t y = tt < 4 ? vw[2 * m + 1].x : vw[2 * m + 1].y;
                    const float2 f = f16x2_to_float2(e4m3x2_to_f16x2(__byte_perm(x, y, sel)));
                    o[m] = bf16x2_rn(f.x * vs[tt], f.y * vs[tt]);
                }
                *reinterpret_cast<uint4*>(vd + (8 * hv + tt) * kF8D + 8 * gv) = make_uint4(o[0], o[1], o[2], o[3]);
            }
            __syncwarp();  // buffer bsel is refilled two pages later
            bsel ^= 1;
        }
    }
}

constexpr size_t kAlign = 1024;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

}  // namespace

Fp8PrefillLayout fp8_prefill_layout(int32_t hkv, int32_t block_size, int32_t max_blocks, int32_t num_chunks,
                                    int64_t max_kv_tokens)
{
    Fp8PrefillLayout L;
    std::memset(&L, 0, sizeof(L));
    if (hkv <= 0 || block_size <= 0 || block_size % 16 || max_blocks <= 0 || num_chunks < 0 || max_kv_tokens < 0)
        return L;
    L.nb = (max_kv_tokens + block_size - 1) / block_size + num_chunks;
    size_t off = 0;
    L.off_first = off;
    off = align_up(off + (size_t)(num_chunks + 1) * 8);
    L.off_owner = off;
    off = align_up(off + (size_t)L.nb * 4);
    L.off_table = off;
    off = align_up(off + (size_t)num_chunks * (size_t)max_blocks * 4);
    const size_t copy = (size_t)L.nb * hkv * block_size * kF8D * 2;
    L.off_k = off;
    off = align_up(off + copy);
    L.off_v = off;
    off = align_up(off + copy);
    L.bytes = off + kAlign;  // slack: the base is aligned up to 1 KB
    return L;
}

kvattn_status launch_prefill_fp8(const PrefillArgs& pa, const void* pool, const Fp8PrefillLayout& L,
                                 void* workspace, cudaStream_t s)
{
    if (pa.num_chunks == 0 || pa.total_q == 0) return KVATTN_OK;
    // launch_prefill's own refusals, checked before anything is launched
    if (L.nb * pa.hkv * pa.block_size >= ((int64_t)1 << 31)) return KVATTN_ERR_UNSUPPORTED;
    if (pa.hq % pa.hkv || (pa.d != 128 && pa.d != 64)) return KVATTN_ERR_UNSUPPORTED;
    if ((int64_t)pa.num_chunks * ((pa.max_q_len + 255) / 256) * pa.hq > 0x7fffffff) return KVATTN_ERR_UNSUPPORTED;
    unsigned char* ws = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(workspace) + kAlign - 1) / kAlign * kAlign);
    Fp8PrefillArgs a;
    std::memset(&a, 0, sizeof(a));
    a.pool = static_cast<const unsigned char*>(pool);
    a.num_blocks = pa.num_blocks;
    a.block_table = pa.block_table;
    a.cu_q_lens = pa.cu_q_lens;
    a.prefix_lens = pa.prefix_lens;
    a.num_chunks = pa.num_chunks;
    a.max_blocks = pa.max_blocks;
    a.max_q_len = pa.max_q_len;
    a.total_q = pa.total_q;
    a.block_size = pa.block_size;
    a.hkv = pa.hkv;
    a.nb = L.nb;
    a.first = reinterpret_cast<int64_t*>(ws + L.off_first);
    a.owner = reinterpret_cast<int32_t*>(ws + L.off_owner);
    a.ctable = reinterpret_cast<int32_t*>(ws + L.off_table);
    a.k_copy = reinterpret_cast<__nv_bfloat16*>(ws + L.off_k);
    a.v_copy = reinterpret_cast<__nv_bfloat16*>(ws + L.off_v);
    a.status = pa.status;
    constexpr int kExpandSmem = kExpandWarps * 2 * kF8Page;
    static SmemLimit limit;
    cudaError_t e = limit.ensure(reinterpret_cast<const void*>(prefill_fp8_expand), kExpandSmem);
    if (e != cudaSuccess) return cuda_status(e);
    int per_sm = 0;  // one wave of resident CTAs (each warp walks a contiguous range of pages)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prefill_fp8_expand, kExpandWarps * 32, kExpandSmem);
    if (e != cudaSuccess) return cuda_status(e);
    e = launch_pdl(prefill_fp8_plan, dim3(1), dim3(1024), 0, s, a);
    if (e != cudaSuccess) return cuda_status(e);
    e = launch_pdl(prefill_fp8_expand, dim3(num_sms() * std::max(1, per_sm)), dim3(kExpandWarps * 32), kExpandSmem, s, a);
    if (e != cudaSuccess) return cuda_status(e);
    PrefillArgs b = pa;
    b.k_pool = a.k_copy;
    b.v_pool = a.v_copy;
    b.block_table = a.ctable;
    b.num_blocks = L.nb;
    return launch_prefill(b, s);
}

}  // namespace kvattn
