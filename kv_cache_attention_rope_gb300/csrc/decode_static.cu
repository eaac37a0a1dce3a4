// kvattn_decode_static_scratch: kvattn_decode for callers that cannot
// allocate device memory.
//
// kvattn_decode needs a caller-provided workspace for the per-chunk partial
// results of the split-KV decode.  Some callers have no way to provide one at
// the point where they run a decode step: an engine that has already handed
// nearly all HBM to its own KV-cache pool and arenas (a cudaMalloc there would
// fail, or fragment memory the engine manages itself), or code running inside
// a host framework's operator interface that exposes no device allocator and
// where calling cudaMalloc/cudaFree itself would synchronise the device in the
// middle of a latency-critical step.  This entry point takes the workspace from
// a fixed-size array in the library's own device memory instead, so it
// allocates nothing.
//
// The array is a file-scope static __device__ object of this translation
// unit's module.  With lazy module loading (the CUDA default) the module, and
// with it the array's 32 MiB, is placed on a device when the first call on
// that device looks up the array's address; from then on the device holds it
// until the process exits.  Host code may not use the array's name as a device
// address (on the host it is only a stand-in symbol), so the address is looked
// up with cudaGetSymbolAddress once per device, with that device current, and
// cached.
#include <cstring>
#include <mutex>

#include "kvattn_internal.cuh"

namespace kvattn {
namespace {

// 32 MiB: the partials of 256 sequences x 32 query heads x 5 chunks of a
// 128-wide head (about 21 MB) fit.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up once;
// the first look-up loads this module onto the device).  nullptr on failure,
// with the failed runtime call's error cleared from cudaGetLastError.
void* static_scratch_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> g(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace kvattn

using namespace kvattn;

extern "C" {

kvattn_status kvattn_decode_static_scratch(const kvattn_config* cfg, const kvattn_cache* cache, const void* q,
                                           const int32_t* block_table, int32_t max_blocks_per_seq,
                                           const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                           int32_t num_splits, void* out, void* stream)
{
    // Set-up form (batch == 0, cache == NULL): place the array on the current
    // device and resolve its address, nothing else.
    if (batch == 0 && !cache) return static_scratch_ptr() ? KVATTN_OK : KVATTN_ERR_CUDA;
    // The argument checks of kvattn_decode, in its order and with its codes;
    // then the size limit of the array, before anything touches the device.
    const kvattn_status st = decode_check(cfg, cache, false, q, block_table, max_blocks_per_seq, seq_lens, batch,
                                          max_seq_len, num_splits, out);
    if (st != KVATTN_OK || batch == 0) return st;
    if (kvattn_decode_workspace_size(cfg, batch, max_seq_len, num_splits) > kStaticScratchBytes)
        return KVATTN_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = static_scratch_ptr();
    if (!scratch) return KVATTN_ERR_CUDA;
    // The partials need no clearing: every slot the combine step reads is
    // written earlier in the same call.
    return kvattn_decode(cfg, cache, q, block_table, max_blocks_per_seq, seq_lens, batch, max_seq_len, num_splits,
                         out, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
