// C ABI of kvattn: argument validation, per-device set-up, dispatch to the
// kernels.  Every check the host can make is made here, before any launch.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kvattn_internal.cuh"

namespace kvattn {

// Module-scope device status word: first device-side error since the last
// kvattn_get_device_status().  One instance per device that loads the module.
__device__ int g_device_status = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

}  // namespace

int* device_status_ptr()
{
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

int num_sms()
{
    const int dev = current_device();
    if (dev < 0) return 1;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

bool device_smem(DeviceSmem* out)
{
    static DeviceSmem cache[kMaxDevices] = {};
    const int dev = current_device();
    if (dev < 0) return false;
    std::lock_guard<std::mutex> g(g_mu);
    DeviceSmem& c = cache[dev];
    if (!c.per_sm) {
        int per_sm = 0, reserved = 0;
        if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            per_sm <= 0)
            return false;
        if (cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
            reserved = 1024;
        c.reserved = reserved;
        c.per_sm = per_sm;
    }
    *out = c;
    return true;
}

cudaError_t SmemLimit::ensure(const void* func, int bytes)
{
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(mu_);
    if (set_[dev] >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) set_[dev] = bytes;
    return e;
}

namespace {

bool config_ok(const kvattn_config* c)
{
    return c && c->num_q_heads > 0 && c->num_kv_heads > 0 && c->head_dim > 0 &&
           (c->dtype == KVATTN_F32 || c->dtype == KVATTN_BF16) && std::isfinite(c->rope_base) &&
           c->rope_base > 0.f && std::isfinite(c->scale) && c->scale >= 0.f;
}

kvattn_status config_supported(const kvattn_config* c)
{
    if (c->num_q_heads % c->num_kv_heads != 0) return KVATTN_ERR_UNSUPPORTED;
    const int g = c->num_q_heads / c->num_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8) return KVATTN_ERR_UNSUPPORTED;
    if (c->head_dim != 64 && c->head_dim != 128) return KVATTN_ERR_UNSUPPORTED;
    return KVATTN_OK;
}

bool cache_ok(const kvattn_cache* k, int32_t max_blocks_per_seq)
{
    if (!k || !k->k_pool || !k->v_pool || k->num_blocks <= 0 || k->num_blocks > INT32_MAX || k->block_size <= 0)
        return false;
    if (max_blocks_per_seq <= 0) return false;
    // a 16-token tile must not cross a block boundary
    if (max_blocks_per_seq > 1 && k->block_size % 16 != 0) return false;
    // 16-byte alignment of the pools (bulk copies)
    if ((reinterpret_cast<uintptr_t>(k->k_pool) | reinterpret_cast<uintptr_t>(k->v_pool)) & 15u) return false;
    return true;
}

float scale_of(const kvattn_config* c)
{
    return c->scale > 0.f ? c->scale : 1.0f / std::sqrt((float)c->head_dim);
}

// Host tables of the rotary embedding for (base, D): per-pair speed in 2^-64
// turns per position, and the float-float cos/sin of k*pi/16, k = 0..4, from
// their nested-radical closed forms (exactly rounded square roots, so the
// values do not depend on the host's libm).
void rope_tables(double base, int d, RopeArgs& a)
{
    static thread_local double cached_base = -1.0;
    static thread_local int cached_d = -1;
    static thread_local uint64_t turns[64];
    if (cached_base != base || cached_d != d) {
        const double two_pi = 6.283185307179586476925286766559;
        for (int i = 0; i < d / 2; ++i) {
            const double f = std::pow(base, -2.0 * (double)i / (double)d) / two_pi;  // turns per position
            turns[i] = (uint64_t)std::llrint(std::ldexp(f, 64));  // f < 1/(2 pi): fits in int64
        }
        cached_base = base;
        cached_d = d;
    }
    std::memcpy(a.turns, turns, sizeof(turns));
    const double r2 = std::sqrt(2.0);
    const double c[5] = {1.0, 0.5 * std::sqrt(2.0 + std::sqrt(2.0 + r2)), 0.5 * std::sqrt(2.0 + r2),
                         0.5 * std::sqrt(2.0 + std::sqrt(2.0 - r2)), 0.5 * r2};
    const double s[5] = {0.0, 0.5 * std::sqrt(2.0 - std::sqrt(2.0 + r2)), 0.5 * std::sqrt(2.0 - r2),
                         0.5 * std::sqrt(2.0 - std::sqrt(2.0 - r2)), 0.5 * r2};
    for (int k = 0; k < 5; ++k) {
        const float ch = (float)c[k], sh = (float)s[k];
        a.sector[k] = make_float4(ch, (float)(c[k] - (double)ch), sh, (float)(s[k] - (double)sh));
    }
}

// One CTA waits on an mbarrier that nothing will complete, through the same
// bounded wait every kernel uses; the wait runs out and records
// KVATTN_ERR_TIMEOUT.
__global__ void selftest_timeout_kernel(int* status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait(&bar, 0, status, limit_ns);
}

}  // namespace

kvattn_status decode_check(const kvattn_config* cfg, const kvattn_cache* cache, bool fp8, const void* q,
                           const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           int32_t batch, int32_t max_seq_len, int32_t num_splits, const void* out)
{
    if (!config_ok(cfg) || batch < 0 || max_seq_len < 0 || num_splits < 0) return KVATTN_ERR_INVALID_ARG;
    kvattn_status st = config_supported(cfg);
    if (st != KVATTN_OK) return st;
    if (!cache_ok(cache, max_blocks_per_seq)) return KVATTN_ERR_INVALID_ARG;
    if (fp8) {
        if (cache->block_size % 16 != 0) return KVATTN_ERR_INVALID_ARG;
        const int g = cfg->num_q_heads / cfg->num_kv_heads;
        if (cfg->dtype != KVATTN_BF16 || cfg->head_dim != 128 || (g != 4 && g != 8)) return KVATTN_ERR_UNSUPPORTED;
    }
    if (batch == 0) return KVATTN_OK;
    if (batch > kMaxDecodeBatch) return KVATTN_ERR_UNSUPPORTED;
    if (!q || !block_table || !seq_lens || !out) return KVATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u) return KVATTN_ERR_INVALID_ARG;
    return KVATTN_OK;
}

}  // namespace kvattn

using namespace kvattn;

extern "C" {

int32_t kvattn_version(void) { return KVATTN_VERSION; }

const char* kvattn_status_string(kvattn_status s)
{
    switch (s) {
        case KVATTN_OK: return "ok";
        case KVATTN_ERR_INVALID_ARG: return "invalid argument";
        case KVATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case KVATTN_ERR_OUT_OF_BLOCKS: return "out of KV blocks";
        case KVATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case KVATTN_ERR_CUDA: return "CUDA error";
        case KVATTN_ERR_TIMEOUT: return "device wait timed out";
        case KVATTN_ERR_BAD_INDEX: return "block id or position out of range";
    }
    return "unknown status";
}

kvattn_status kvattn_rope_append(const kvattn_config* cfg, const kvattn_cache* cache, void* q, const void* k,
                                 const void* v, const int32_t* positions, const int32_t* seq_ids,
                                 const int32_t* block_table, int32_t num_seqs, int32_t max_blocks_per_seq,
                                 int32_t num_tokens, void* stream)
{
    if (!config_ok(cfg)) return KVATTN_ERR_INVALID_ARG;
    const int64_t qrow = (int64_t)cfg->num_q_heads * cfg->head_dim;
    const int64_t kvrow = (int64_t)cfg->num_kv_heads * cfg->head_dim;
    return kvattn_rope_append_strided(cfg, cache, q, qrow, k, kvrow, v, kvrow, nullptr, positions, seq_ids,
                                      block_table, num_seqs, max_blocks_per_seq, num_tokens, stream);
}

kvattn_status kvattn_rope_append_strided(const kvattn_config* cfg, const kvattn_cache* cache, void* q,
                                         int64_t q_stride, const void* k, int64_t k_stride, const void* v,
                                         int64_t v_stride, void* q_out, const int32_t* positions,
                                         const int32_t* seq_ids, const int32_t* block_table, int32_t num_seqs,
                                         int32_t max_blocks_per_seq, int32_t num_tokens, void* stream)
{
    if (!config_ok(cfg) || num_tokens < 0 || num_seqs <= 0) return KVATTN_ERR_INVALID_ARG;
    kvattn_status st = config_supported(cfg);
    if (st != KVATTN_OK) return st;
    if (!cache_ok(cache, max_blocks_per_seq)) return KVATTN_ERR_INVALID_ARG;
    // a row never overlaps the next one, and every row starts on a 16-byte boundary
    const int64_t e = cfg->dtype == KVATTN_BF16 ? 2 : 4;
    const int64_t qrow = (int64_t)cfg->num_q_heads * cfg->head_dim;
    const int64_t kvrow = (int64_t)cfg->num_kv_heads * cfg->head_dim;
    const int64_t max_stride = INT64_MAX / 4 / std::max<int64_t>(1, num_tokens);
    if (q_stride < qrow || k_stride < kvrow || v_stride < kvrow) return KVATTN_ERR_INVALID_ARG;
    if (q_stride > max_stride || k_stride > max_stride || v_stride > max_stride) return KVATTN_ERR_INVALID_ARG;
    if (((q_stride | k_stride | v_stride) * e) & 15) return KVATTN_ERR_INVALID_ARG;
    if (num_tokens == 0) return KVATTN_OK;
    if (!q || !k || !v || !positions || !seq_ids || !block_table) return KVATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(q_out)) & 15u)
        return KVATTN_ERR_INVALID_ARG;
    RopeArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = q;
    a.k = k;
    a.v = v;
    a.q_stride = q_stride * e;
    a.k_stride = k_stride * e;
    a.v_stride = v_stride * e;
    a.q_out = q_out ? q_out : q;
    a.q_out_stride = q_out ? qrow * e : a.q_stride;
    a.k_pool = cache->k_pool;
    a.v_pool = cache->v_pool;
    a.positions = positions;
    a.seq_ids = seq_ids;
    a.block_table = block_table;
    a.num_blocks = cache->num_blocks;
    a.block_size = cache->block_size;
    a.num_seqs = num_seqs;
    a.max_blocks = max_blocks_per_seq;
    a.num_tokens = num_tokens;
    a.hq = cfg->num_q_heads;
    a.hkv = cfg->num_kv_heads;
    a.d = cfg->head_dim;
    a.dtype = cfg->dtype;
    a.status = device_status_ptr();
    if (!a.status) return KVATTN_ERR_CUDA;
    rope_tables((double)cfg->rope_base, cfg->head_dim, a);
    return launch_rope_append(a, static_cast<cudaStream_t>(stream));
}

namespace {

// bytes of one layer's K (or V) region, 0 if invalid or too large
int64_t layer_region_bytes(const kvattn_config* cfg, int32_t num_layers, int64_t num_blocks, int32_t block_size)
{
    if (!config_ok(cfg) || num_layers <= 0 || num_blocks <= 0 || block_size <= 0) return 0;
    const int64_t e = cfg->dtype == KVATTN_BF16 ? 2 : 4;
    const int64_t per_block = (int64_t)cfg->num_kv_heads * block_size * cfg->head_dim * e;
    if (per_block <= 0 || num_blocks > INT64_MAX / 4 / per_block / (2 * (int64_t)num_layers)) return 0;
    return num_blocks * per_block;
}

}  // namespace

size_t kvattn_layered_cache_bytes(const kvattn_config* cfg, int32_t num_layers, int64_t num_blocks,
                                  int32_t block_size)
{
    const int64_t region = layer_region_bytes(cfg, num_layers, num_blocks, block_size);
    return region ? (size_t)(region * 2 * num_layers) : 0;
}

kvattn_status kvattn_layer_cache(const kvattn_config* cfg, void* base, int32_t num_layers, int64_t num_blocks,
                                 int32_t block_size, int32_t layer, kvattn_cache* out)
{
    if (!out || !base || layer < 0 || layer >= num_layers) return KVATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0) return KVATTN_ERR_INVALID_ARG;
    const int64_t region = layer_region_bytes(cfg, num_layers, num_blocks, block_size);
    if (!region) return KVATTN_ERR_INVALID_ARG;
    const kvattn_status st = config_supported(cfg);
    if (st != KVATTN_OK) return st;
    char* b = static_cast<char*>(base);
    out->k_pool = b + (2 * (int64_t)layer) * region;
    out->v_pool = b + (2 * (int64_t)layer + 1) * region;
    out->num_blocks = num_blocks;
    out->block_size = block_size;
    return KVATTN_OK;
}

namespace {

kvattn_status copy_blocks(const kvattn_config* cfg, char* k_base, char* v_base, int64_t layer_stride,
                          int32_t layers, int64_t num_blocks, int32_t block_size, const int32_t* src_ids,
                          const int32_t* dst_ids, int32_t n, void* stream)
{
    if (n < 0) return KVATTN_ERR_INVALID_ARG;
    if (n == 0) return KVATTN_OK;
    if (!src_ids || !dst_ids) return KVATTN_ERR_INVALID_ARG;
    CopyArgs a;
    std::memset(&a, 0, sizeof(a));
    a.k_base = k_base;
    a.v_base = v_base;
    a.layer_stride = layer_stride;
    a.layers = layers;
    a.block_bytes = (int64_t)cfg->num_kv_heads * block_size * cfg->head_dim * (cfg->dtype == KVATTN_BF16 ? 2 : 4);
    a.num_blocks = num_blocks;
    a.src = src_ids;
    a.dst = dst_ids;
    a.n = n;
    a.status = device_status_ptr();
    if (!a.status) return KVATTN_ERR_CUDA;
    return launch_copy_blocks(a, static_cast<cudaStream_t>(stream));
}

}  // namespace

kvattn_status kvattn_copy_blocks(const kvattn_config* cfg, const kvattn_cache* cache, const int32_t* src_ids,
                                 const int32_t* dst_ids, int32_t n, void* stream)
{
    if (!config_ok(cfg) || !cache_ok(cache, 1)) return KVATTN_ERR_INVALID_ARG;
    const kvattn_status st = config_supported(cfg);
    if (st != KVATTN_OK) return st;
    return copy_blocks(cfg, static_cast<char*>(cache->k_pool), static_cast<char*>(cache->v_pool), 0, 1,
                       cache->num_blocks, cache->block_size, src_ids, dst_ids, n, stream);
}

kvattn_status kvattn_copy_blocks_layered(const kvattn_config* cfg, void* base, int32_t num_layers,
                                         int64_t num_blocks, int32_t block_size, const int32_t* src_ids,
                                         const int32_t* dst_ids, int32_t n, void* stream)
{
    kvattn_cache first;
    const kvattn_status st = kvattn_layer_cache(cfg, base, num_layers, num_blocks, block_size, 0, &first);
    if (st != KVATTN_OK) return st;
    if (num_blocks > INT32_MAX) return KVATTN_ERR_INVALID_ARG;
    const int64_t region = static_cast<char*>(first.v_pool) - static_cast<char*>(first.k_pool);
    return copy_blocks(cfg, static_cast<char*>(first.k_pool), static_cast<char*>(first.v_pool), 2 * region,
                       num_layers, num_blocks, block_size, src_ids, dst_ids, n, stream);
}

int32_t kvattn_decode_num_splits(const kvattn_config* cfg, int32_t batch, int32_t max_seq_len, int32_t num_splits)
{
    if (!config_ok(cfg) || config_supported(cfg) != KVATTN_OK || batch < 0 || max_seq_len < 0 || num_splits < 0)
        return 0;
    return decode_plan(batch, cfg->num_kv_heads, cfg->num_q_heads / cfg->num_kv_heads, max_seq_len, num_splits)
        .slots;
}

namespace {
// Workspace: [batch][segments] int32 piece counts | [batch][hq][slots][D] f32
// partial outputs | [batch][hq][slots][2] f32 (max, sum); each 256-byte aligned.
struct WorkspaceLayout {
    size_t nslots_off, o_off, ml_off, bytes;
};
WorkspaceLayout workspace_layout(const kvattn_config* cfg, int32_t batch, int32_t slots)
{
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    WorkspaceLayout w;
    const size_t rows = (size_t)batch * cfg->num_q_heads * slots;
    w.nslots_off = 0;
    w.o_off = up((size_t)batch * decode_segments(cfg->num_q_heads, cfg->num_kv_heads) * 4);
    w.ml_off = w.o_off + up(rows * cfg->head_dim * 4);
    w.bytes = std::max<size_t>(256, w.ml_off + up(rows * 2 * 4));
    return w;
}
}  // namespace

size_t kvattn_decode_workspace_size(const kvattn_config* cfg, int32_t batch, int32_t max_seq_len,
                                    int32_t num_splits)
{
    const int32_t slots = kvattn_decode_num_splits(cfg, batch, max_seq_len, num_splits);
    if (slots <= 0) return 0;
    return workspace_layout(cfg, batch, slots).bytes;
}

namespace {

kvattn_status decode_any(const kvattn_config* cfg, const kvattn_cache* cache, bool fp8,
                         const void* q, const int32_t* block_table, int32_t max_blocks_per_seq,
                         const int32_t* seq_lens, int32_t batch, int32_t max_seq_len, int32_t num_splits, void* out,
                         void* workspace, size_t workspace_bytes, void* stream)
{
    const kvattn_status st = decode_check(cfg, cache, fp8, q, block_table, max_blocks_per_seq, seq_lens, batch,
                                          max_seq_len, num_splits, out);
    if (st != KVATTN_OK || batch == 0) return st;
    const DecodePlan p = decode_plan(batch, cfg->num_kv_heads, cfg->num_q_heads / cfg->num_kv_heads, max_seq_len,
                                     num_splits);
    const WorkspaceLayout wl = workspace_layout(cfg, batch, p.slots);
    if (p.slots > 1) {
        if (!workspace || workspace_bytes < wl.bytes) return KVATTN_ERR_WORKSPACE_TOO_SMALL;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return KVATTN_ERR_INVALID_ARG;
    }
    DecodeArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = q;
    a.k_pool = cache->k_pool;
    a.v_pool = cache->v_pool;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.out = out;
    if (p.slots > 1) {
        char* w = static_cast<char*>(workspace);
        a.nslots = reinterpret_cast<int32_t*>(w + wl.nslots_off);
        a.part_o = reinterpret_cast<float*>(w + wl.o_off);
        a.part_ml = reinterpret_cast<float*>(w + wl.ml_off);
    }
    a.num_blocks = cache->num_blocks;
    a.block_size = cache->block_size;
    a.max_blocks = max_blocks_per_seq;
    a.batch = batch;
    a.max_seq_len = max_seq_len;
    a.splits = p.slots;
    a.hq = cfg->num_q_heads;
    a.hkv = cfg->num_kv_heads;
    a.d = cfg->head_dim;
    a.dtype = cfg->dtype;
    a.scale_log2 = scale_of(cfg) * 1.4426950408889634f;
    a.fp8 = fp8 ? 1 : 0;
    a.status = device_status_ptr();
    if (!a.status) return KVATTN_ERR_CUDA;
    return launch_decode(a, static_cast<cudaStream_t>(stream));
}

}  // namespace

kvattn_status kvattn_decode(const kvattn_config* cfg, const kvattn_cache* cache, const void* q,
                            const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                            int32_t batch, int32_t max_seq_len, int32_t num_splits, void* out, void* workspace,
                            size_t workspace_bytes, void* stream)
{
    return decode_any(cfg, cache, false, q, block_table, max_blocks_per_seq, seq_lens, batch, max_seq_len,
                      num_splits, out, workspace, workspace_bytes, stream);
}

kvattn_status kvattn_decode_fp8(const kvattn_config* cfg, const kvattn_cache_fp8* cache, const void* q,
                                const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                int32_t batch, int32_t max_seq_len, int32_t num_splits, void* out, void* workspace,
                                size_t workspace_bytes, void* stream)
{
    if (!cache) return KVATTN_ERR_INVALID_ARG;
    const kvattn_cache c{cache->pool, cache->pool, cache->num_blocks, cache->block_size};
    return decode_any(cfg, &c, true, q, block_table, max_blocks_per_seq, seq_lens, batch, max_seq_len, num_splits,
                      out, workspace, workspace_bytes, stream);
}

kvattn_status kvattn_rope_append_fp8(const kvattn_config* cfg, const kvattn_cache_fp8* cache, void* q,
                                     const void* k, const void* v, const int32_t* positions, const int32_t* seq_ids,
                                     const int32_t* block_table, int32_t num_seqs, int32_t max_blocks_per_seq,
                                     int32_t num_tokens, void* stream)
{
    if (!config_ok(cfg) || num_tokens < 0 || num_seqs <= 0 || !cache) return KVATTN_ERR_INVALID_ARG;
    kvattn_status st = config_supported(cfg);
    if (st != KVATTN_OK) return st;
    if (cfg->dtype != KVATTN_BF16 || cfg->head_dim != 128) return KVATTN_ERR_UNSUPPORTED;
    const kvattn_cache c{cache->pool, cache->pool, cache->num_blocks, cache->block_size};
    if (!cache_ok(&c, max_blocks_per_seq) || cache->block_size % 16 != 0) return KVATTN_ERR_INVALID_ARG;
    if (num_tokens == 0) return KVATTN_OK;
    if (!q || !k || !v || !positions || !seq_ids || !block_table) return KVATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u)
        return KVATTN_ERR_INVALID_ARG;
    RopeArgs a;
    std::memset(&a, 0, sizeof(a));
    const int64_t qrow = (int64_t)cfg->num_q_heads * cfg->head_dim * 2;
    const int64_t kvrow = (int64_t)cfg->num_kv_heads * cfg->head_dim * 2;
    a.q = q;
    a.k = k;
    a.v = v;
    a.q_stride = qrow;
    a.k_stride = kvrow;
    a.v_stride = kvrow;
    a.q_out = q;
    a.q_out_stride = qrow;
    a.k_pool = cache->pool;
    a.v_pool = cache->pool;
    a.fp8 = 1;
    a.positions = positions;
    a.seq_ids = seq_ids;
    a.block_table = block_table;
    a.num_blocks = cache->num_blocks;
    a.block_size = cache->block_size;
    a.num_seqs = num_seqs;
    a.max_blocks = max_blocks_per_seq;
    a.num_tokens = num_tokens;
    a.hq = cfg->num_q_heads;
    a.hkv = cfg->num_kv_heads;
    a.d = cfg->head_dim;
    a.dtype = cfg->dtype;
    a.status = device_status_ptr();
    if (!a.status) return KVATTN_ERR_CUDA;
    rope_tables((double)cfg->rope_base, cfg->head_dim, a);
    return launch_rope_append_fp8(a, static_cast<cudaStream_t>(stream));
}

kvattn_status kvattn_prefill_chunk(const kvattn_config* cfg, const kvattn_cache* cache, const void* q,
                                   const int32_t* cu_q_lens, const int32_t* prefix_lens,
                                   const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_chunks,
                                   int32_t max_q_len, int32_t total_q, void* out, void* stream)
{
    if (!config_ok(cfg) || num_chunks < 0 || max_q_len < 0 || total_q < 0) return KVATTN_ERR_INVALID_ARG;
    kvattn_status st = config_supported(cfg);
    if (st != KVATTN_OK) return st;
    if (cfg->dtype != KVATTN_BF16 || (cfg->head_dim != 128 && cfg->head_dim != 64)) return KVATTN_ERR_UNSUPPORTED;
    if (!cache_ok(cache, max_blocks_per_seq)) return KVATTN_ERR_INVALID_ARG;
    if (cache->block_size % 16 != 0) return KVATTN_ERR_UNSUPPORTED;
    if (num_chunks == 0 || total_q == 0) return KVATTN_OK;
    if (!q || !cu_q_lens || !prefix_lens || !block_table || !out) return KVATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u) return KVATTN_ERR_INVALID_ARG;
    PrefillArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = q;
    a.k_pool = cache->k_pool;
    a.v_pool = cache->v_pool;
    a.cu_q_lens = cu_q_lens;
    a.prefix_lens = prefix_lens;
    a.block_table = block_table;
    a.out = out;
    a.num_blocks = cache->num_blocks;
    a.block_size = cache->block_size;
    a.max_blocks = max_blocks_per_seq;
    a.num_chunks = num_chunks;
    a.max_q_len = max_q_len;
    a.total_q = total_q;
    a.hq = cfg->num_q_heads;
    a.hkv = cfg->num_kv_heads;
    a.d = cfg->head_dim;
    a.scale_log2 = scale_of(cfg) * 1.4426950408889634f;
    a.status = device_status_ptr();
    if (!a.status) return KVATTN_ERR_CUDA;
    return launch_prefill(a, static_cast<cudaStream_t>(stream));
}

size_t kvattn_prefill_fp8_workspace_size(const kvattn_config* cfg, int32_t block_size, int32_t max_blocks_per_seq,
                                         int32_t num_chunks, int64_t max_kv_tokens)
{
    if (!config_ok(cfg) || config_supported(cfg) != KVATTN_OK) return 0;
    if (cfg->dtype != KVATTN_BF16 || cfg->head_dim != 128) return 0;
    return fp8_prefill_layout(cfg->num_kv_heads, block_size, max_blocks_per_seq, num_chunks, max_kv_tokens).bytes;
}

kvattn_status kvattn_prefill_chunk_fp8(const kvattn_config* cfg, const kvattn_cache_fp8* cache, const void* q,
                                       const int32_t* cu_q_lens, const int32_t* prefix_lens,
                                       const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_chunks,
                                       int32_t max_q_len, int32_t total_q, int64_t max_kv_tokens, void* out,
                                       void* workspace, size_t workspace_bytes, void* stream)
{
    if (!config_ok(cfg) || num_chunks < 0 || max_q_len < 0 || total_q < 0 || max_kv_tokens < 0 || !cache)
        return KVATTN_ERR_INVALID_ARG;
    kvattn_status st = config_supported(cfg);
    if (st != KVATTN_OK) return st;
    if (cfg->dtype != KVATTN_BF16 || cfg->head_dim != 128) return KVATTN_ERR_UNSUPPORTED;
    const kvattn_cache c{cache->pool, cache->pool, cache->num_blocks, cache->block_size};
    if (!cache_ok(&c, max_blocks_per_seq) || cache->block_size % 16 != 0) return KVATTN_ERR_INVALID_ARG;
    if (num_chunks == 0 || total_q == 0) return KVATTN_OK;
    if (!q || !cu_q_lens || !prefix_lens || !block_table || !out || !workspace) return KVATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u) return KVATTN_ERR_INVALID_ARG;
    const Fp8PrefillLayout L =
        fp8_prefill_layout(cfg->num_kv_heads, cache->block_size, max_blocks_per_seq, num_chunks, max_kv_tokens);
    if (L.bytes == 0) return KVATTN_ERR_INVALID_ARG;
    if (workspace_bytes < L.bytes) return KVATTN_ERR_WORKSPACE_TOO_SMALL;
    PrefillArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = q;
    a.cu_q_lens = cu_q_lens;
    a.prefix_lens = prefix_lens;
    a.block_table = block_table;
    a.out = out;
    a.num_blocks = cache->num_blocks;
    a.block_size = cache->block_size;
    a.max_blocks = max_blocks_per_seq;
    a.num_chunks = num_chunks;
    a.max_q_len = max_q_len;
    a.total_q = total_q;
    a.hq = cfg->num_q_heads;
    a.hkv = cfg->num_kv_heads;
    a.d = cfg->head_dim;
    a.scale_log2 = scale_of(cfg) * 1.4426950408889634f;
    a.status = device_status_ptr();
    if (!a.status) return KVATTN_ERR_CUDA;
    return launch_prefill_fp8(a, cache->pool, L, workspace, static_cast<cudaStream_t>(stream));
}

kvattn_status kvattn_selftest_wait_timeout(int32_t limit_us, void* stream)
{
    if (limit_us < 1 || limit_us > 1000000) return KVATTN_ERR_INVALID_ARG;
    int* st = device_status_ptr();
    if (!st) return KVATTN_ERR_CUDA;
    selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st, (uint64_t)limit_us * 1000ull);
    return cuda_status(cudaGetLastError());
}

kvattn_status kvattn_get_device_status(void* stream, int32_t* out)
{
    if (!out) return KVATTN_ERR_INVALID_ARG;
    int* p = device_status_ptr();
    if (!p) return KVATTN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVATTN_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KVATTN_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return KVATTN_ERR_CUDA;
    *out = v;
    return KVATTN_OK;
}

}  // extern "C"
