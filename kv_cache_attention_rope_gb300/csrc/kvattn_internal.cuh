// Internal declarations shared by the kvattn CUDA translation units:
// launch entry points, device status reporting, and thin inline-PTX wrappers
// for the sm_100-family asynchronous machinery (mbarrier, bulk copies,
// tcgen05).  Everything here is written from the public PTX ISA description.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kvattn.h"

namespace kvattn {

// ---------------------------------------------------------------- host side

// Device status word of the current device (a module-scope __device__ int).
int* device_status_ptr();

// One-line CUDA error mapping.
inline kvattn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVATTN_OK : KVATTN_ERR_CUDA; }

// Kernel launches with programmatic stream serialization: a kernel may be
// scheduled while the kernel before it on the stream drains, which hides the
// launch gap between the step's kernels.  Every kernel so launched starts
// with pdl_wait(), which returns once the previous grid has completed and its
// memory operations are visible, so stream order holds for every global
// access (and a kernel launched without the attribute returns at once).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

int num_sms();

// Shared-memory figures of the current device (cached per device).
struct DeviceSmem {
    int per_sm;          // cudaDevAttrMaxSharedMemoryPerMultiprocessor
    int reserved;        // cudaDevAttrReservedSharedMemoryPerBlock
};
bool device_smem(DeviceSmem* out);

// A kernel's dynamic shared-memory limit is a per-device attribute: raise it
// to at least `bytes` on the current device, once per (kernel, device, size).
class SmemLimit {
public:
    cudaError_t ensure(const void* func, int bytes);

private:
    std::mutex mu_;
    int set_[64] = {};
};

struct RopeArgs {
    void* q;
    const void* k;
    const void* v;
    int64_t q_stride, k_stride, v_stride;  // bytes from one token's row to the next
    void* q_out;                           // rotated q rows (== q: in place)
    int64_t q_out_stride;                  // bytes
    int32_t fp8;  // k_pool is an fp8 page pool (v_pool unused)
    void* k_pool;
    void* v_pool;
    const int32_t* positions;
    const int32_t* seq_ids;
    const int32_t* block_table;
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_seqs;
    int32_t max_blocks;
    int32_t num_tokens;
    int32_t hq, hkv, d;
    int32_t dtype;
    int* status;
    // per-pair rotation speed in turns per position, 2^-64 fixed point:
    // round(base^(-2i/D) / (2 pi) * 2^64)
    uint64_t turns[64];
    // cos/sin of k*pi/16, k = 0..4, as float-float pairs (c_hi, c_lo, s_hi, s_lo)
    float4 sector[5];
};
kvattn_status launch_rope_append(const RopeArgs& a, cudaStream_t s);
kvattn_status launch_rope_append_fp8(const RopeArgs& a, cudaStream_t s);  // a.fp8 set

// fp8 cache page: the 16 tokens of one (block, KV head, 16-token group) at
// D = 128, laid out for the decode kernel (one bulk copy per page, every
// fragment load conflict-free):
//   [0, 2048)     K codes, token r: 16-byte chunk c (dims 16c..16c+15) at
//                 r * 128 + 16 * (c ^ f8_swz(r))
//   [2048, 4096)  V codes transposed: dim d, token r at 2048 + 16 * d + r
//   [4096, 4160)  K scales, fp32 [16];  [4160, 4224) V scales, fp32 [16]
constexpr int kF8Page = 4224, kF8VOff = 2048, kF8KsOff = 4096, kF8VsOff = 4160;
__host__ __device__ constexpr int f8_swz(int r) { return (r & 1) | ((r >> 1) & 6); }

// Whole-block copies over every K/V region of a (multi-layer) cache: region
// r = 2 * layer + (0: K, 1: V) starts at (r odd ? v_base : k_base) +
// layer * layer_stride.
struct CopyArgs {
    char* k_base;
    char* v_base;
    int64_t layer_stride;   // bytes; 0 for one layer
    int64_t block_bytes;    // Hkv * block_size * D * element size (a multiple of 16)
    int64_t num_blocks;
    const int32_t* src;
    const int32_t* dst;
    int32_t n;
    int32_t layers;
    int* status;
};
kvattn_status launch_copy_blocks(const CopyArgs& a, cudaStream_t s);

struct DecodeArgs {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* block_table;
    const int32_t* seq_lens;
    void* out;
    int32_t fp8;  // k_pool is an fp8 page pool (v_pool unused)
    int32_t* nslots;   // [batch][segments]: pieces each segment was cut into
    float* part_o;     // [batch][hq][splits][d]
    float* part_ml;    // [batch][hq][splits][2] (max in log2 units, sum)
    int64_t num_blocks;
    int32_t block_size;
    int32_t max_blocks;
    int32_t batch;
    int32_t max_seq_len;
    int32_t splits;    // most pieces per segment (plan.slots); 1 = whole segments
    int32_t hq, hkv, d;
    int32_t dtype;
    float scale_log2;  // softmax scale * log2(e)
    int* status;
};
kvattn_status launch_decode(const DecodeArgs& a, cudaStream_t s);

// Largest decode batch (the kernels keep a per-sequence prefix sum in shared memory).
constexpr int32_t kMaxDecodeBatch = 8192;

// Every host-side check of kvattn_decode / kvattn_decode_fp8 that does not
// involve the workspace, in their order (the same status codes).
kvattn_status decode_check(const kvattn_config* cfg, const kvattn_cache* cache, bool fp8, const void* q,
                           const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           int32_t batch, int32_t max_seq_len, int32_t num_splits, const void* out);

// Most pieces a (sequence, KV head) segment may be cut into.  splits > 0 is
// the caller's cap; 0 lets the library choose.  1 = every segment whole.
struct DecodePlan {
    int32_t slots;
};
DecodePlan decode_plan(int32_t batch, int32_t hkv, int32_t group, int32_t max_seq_len, int32_t splits);

// Segments per sequence, at most: KV heads, times 2 when a GQA group of 8 is
// split into two segments of 4 query heads (the CUDA-core path: fp32 caches
// or D = 64; the tensor-core path keeps a group of 8 in one segment).  Sizes
// the workspace's piece counts.
inline int32_t decode_segments(int32_t hq, int32_t hkv)
{
    const int32_t g = hq / hkv;
    return hkv * (g > 4 ? g / 4 : 1);
}

struct PrefillArgs {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* cu_q_lens;
    const int32_t* prefix_lens;
    const int32_t* block_table;
    void* out;
    int64_t num_blocks;
    int32_t block_size;
    int32_t max_blocks;
    int32_t num_chunks;
    int32_t max_q_len;
    int32_t total_q;
    int32_t hq, hkv, d;
    float scale_log2;
    int* status;
};
kvattn_status launch_prefill(const PrefillArgs& a, cudaStream_t s);

// Workspace of the fp8 prefill: the chunks' blocks expanded to bf16 (nb
// blocks, K and V), their block table, owners and first blocks.  bytes == 0
// for invalid arguments.
struct Fp8PrefillLayout {
    int64_t nb;
    size_t off_first, off_owner, off_table, off_k, off_v, bytes;
};
Fp8PrefillLayout fp8_prefill_layout(int32_t hkv, int32_t block_size, int32_t max_blocks, int32_t num_chunks,
                                    int64_t max_kv_tokens);
// Expands the chunks' fp8 pages into the workspace, then runs launch_prefill
// over the bf16 copy (pa's pools and table are replaced).
kvattn_status launch_prefill_fp8(const PrefillArgs& pa, const void* pool, const Fp8PrefillLayout& L,
                                 void* workspace, cudaStream_t s);

// ---------------------------------------------------------------- device side

// Waits for the grid launched before this one on the stream (see launch_pdl).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// First error wins; later ones are dropped.
__device__ __forceinline__ void record_error(int* status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// mbarrier (shared::cta) --------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait limit of every bounded wait: a legitimate wait here is microseconds.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// Bounded phase wait.  Returns false (and records KVATTN_ERR_TIMEOUT) if the
// phase with the given parity has not completed within limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            record_error(status, KVATTN_ERR_TIMEOUT);
            return false;
        }
    }
}

// Bulk (non-tensor) asynchronous copy global -> shared, completion counted
// in bytes on `bar`.  Both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// L2 policy for data read once (streamed KV pages).
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// packed f32x2 math (sm_100 family: one instruction for two lanes' worth of
// fp32 work; the pair lives in one 64-bit register, element 0 in the low half)

__device__ __forceinline__ uint64_t pk(float lo, float hi)
{
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float pk_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float pk_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// bf16 <-> fp32 on raw bits -----------------------------------------------

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16_rn(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace kvattn
