/*
 * kvattn.h -- C ABI of the RoPE + KV-cache + attention hot path of an LLM
 * inference step, for one NVIDIA GB300 (sm_103a) GPU.
 *
 * The operations follow the problem statement of a set of web tutorials on
 * hand-writing an LLM inference engine (cited per function below by page
 * title and section):
 *   [RoPE page]    "Hand-writing an LLM inference engine: Tokenizer, KV Cache
 *                  and RoPE"
 *   [Engine page]  "From-scratch AI inference engine: beyond calling packages"
 *   [Nano-vLLM]    "Understanding an LLM inference engine through Nano-vLLM,
 *                  Part 2"
 *   [Series intro] "Hand-writing an LLM inference engine", chapter 1
 *
 * Conventions shared by every call
 *   - Pointers documented "device" are CUDA device pointers owned by the
 *     caller; the library never allocates, frees or retains device memory
 *     (the exceptions are module-scope device variables: a 4-byte status
 *     word, and the 32 MiB split scratch of kvattn_decode_static_scratch).
 *   - Per-device state (those variables' addresses, kernel attributes,
 *     tensor maps) is set up on first use with the device current and then
 *     cached; it is not valid after cudaDeviceReset on that device.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  GPU calls are asynchronous on that stream; a returned
 *     KVATTN_OK means the work was validated and launched.
 *   - Every argument the host can check is checked before anything is
 *     launched; a failed check returns an error and launches nothing.
 *   - Index errors only the GPU can see (a block id outside the pool, a
 *     position past the block table) make the kernel skip that access and
 *     record KVATTN_ERR_BAD_INDEX in the device status word; a bounded wait
 *     that runs out records KVATTN_ERR_TIMEOUT.  Read and clear it with
 *     kvattn_get_device_status().
 *   - Element type: KVATTN_F32 or KVATTN_BF16 for q, k, v, the cache and the
 *     output alike; arithmetic is fp32 with fp32 accumulation.
 *   - Supported: head_dim 64 or 128, num_q_heads % num_kv_heads == 0 with
 *     group size G = num_q_heads / num_kv_heads in {1, 2, 4, 8}.  Query head
 *     j reads KV head j / G (contiguous groups).  Anything else returns
 *     KVATTN_ERR_UNSUPPORTED.
 *
 * KV cache layout (one layer; K and V are separate pools):
 *   k_pool, v_pool: [num_blocks][num_kv_heads][block_size][head_dim]
 *   Token position p of the sequence owning block-table row r lives in block
 *   b = block_table[r * max_blocks_per_seq + p / block_size] at offset
 *   p % block_size ([Nano-vLLM], section 05: physical block from the table,
 *   offset inside the block).  A paged cache uses block_size = 16; a
 *   contiguous cache is the same layout with block_size = max_len and one
 *   table column holding the row of each sequence ([Engine page],
 *   section 3.2: contiguous per-sequence preallocation vs fixed-size pages).
 *   block_size must be a multiple of 16 when max_blocks_per_seq > 1.
 */
#ifndef KVATTN_H
#define KVATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVATTN_VERSION 1

typedef enum {
    KVATTN_OK = 0,
    KVATTN_ERR_INVALID_ARG = 1,      /* null pointer, negative size, bad id ... */
    KVATTN_ERR_UNSUPPORTED = 2,      /* head_dim / group size / dtype not built */
    KVATTN_ERR_OUT_OF_BLOCKS = 3,    /* allocator exhausted (nothing allocated) */
    KVATTN_ERR_WORKSPACE_TOO_SMALL = 4,
    KVATTN_ERR_CUDA = 5,             /* a CUDA runtime call or launch failed */
    KVATTN_ERR_TIMEOUT = 6,          /* device: a bounded wait ran out */
    KVATTN_ERR_BAD_INDEX = 7         /* device: block id / position out of range */
} kvattn_status;

typedef enum { KVATTN_F32 = 0, KVATTN_BF16 = 1 } kvattn_dtype;

typedef struct {
    int32_t num_q_heads;   /* Hq */
    int32_t num_kv_heads;  /* Hkv; Hq % Hkv == 0 */
    int32_t head_dim;      /* D: 64 or 128 */
    int32_t dtype;         /* kvattn_dtype */
    float rope_base;       /* theta_i = rope_base^(-2i/D); 10000 on the pages */
    float scale;           /* softmax scale; 0 => 1/sqrt(head_dim) */
} kvattn_config;

typedef struct {
    void* k_pool;          /* device, [num_blocks][Hkv][block_size][D] */
    void* v_pool;          /* device, same shape */
    int64_t num_blocks;
    int32_t block_size;
} kvattn_cache;

/*
 * FP8 KV cache (e4m3 codes, 1 byte per element) with one fp32 scale per
 * (slot, KV head): the value of element d of head h at slot t is
 * code[t][h][d] * scale[t][h].  D = 128 only.
 *
 * One pool holds K, V and their scales in pages of 16 tokens:
 *   pool: [num_blocks][Hkv][block_size / 16][4224 bytes]
 * Page of tokens r = 0..15 (positions 16j + r of the block's group j):
 *   [0, 2048)     K codes: token r's 16-byte chunk c (dims 16c .. 16c+15)
 *                 at byte r*128 + 16*(c ^ s(r)),  s(r) = (r & 1) | ((r >> 1) & 6)
 *   [2048, 4096)  V codes, transposed: dim d of token r at byte 2048 + 16*d + r
 *   [4096, 4160)  K scales, fp32 [16]
 *   [4160, 4224)  V scales, fp32 [16]
 * The decode kernel fetches one page per (16 tokens, KV head) with a single
 * bulk copy; the chunk rotation and the transposed V make every operand
 * fragment a conflict-free 32-bit shared-memory load.
 */
typedef struct {
    void* pool;            /* device, 16-byte aligned, num_blocks*Hkv*(block_size/16)*4224 bytes */
    int64_t num_blocks;
    int32_t block_size;    /* a multiple of 16 */
} kvattn_cache_fp8;

/* Library version (KVATTN_VERSION) and a static string for a status code. */
int32_t kvattn_version(void);
const char* kvattn_status_string(kvattn_status s);

/*
 * kvattn_rope_append -- rotary position embedding of the new tokens' q and k,
 * fused with writing k (rotated) and v (as given) into the cache.
 *
 * [RoPE page], section 4: vector split into adjacent pairs (x0,x1),(x2,x3),...
 * and pair i rotated by the 2-D rotation of angle m*theta_i,
 * theta_i = rope_base^(-2i/D), m = the token's position:
 *     x'[2i]   = x[2i] cos(m theta_i) - x[2i+1] sin(m theta_i)
 *     x'[2i+1] = x[2i] sin(m theta_i) + x[2i+1] cos(m theta_i)
 * [Engine page], section 3.2: the new token's K and V are written at the
 * cache index equal to its absolute position, which is also the RoPE
 * position.  v is not rotated ([Series intro], section 2.2: RoPE rotates Q
 * and K).
 *
 *   q           device, [num_tokens][Hq][D], rotated IN PLACE
 *   k, v        device, [num_tokens][Hkv][D], read only
 *   positions   device, [num_tokens] int32, absolute position of each token
 *   seq_ids     device, [num_tokens] int32, block-table row of each token
 *   block_table device, [num_seqs][max_blocks_per_seq] int32
 * Each stored element is the round-to-nearest-even of the rotation of the
 * input values.  Tokens may belong to any rows, in any order; two tokens must
 * not name the same (row, position).
 * Errors: INVALID_ARG (null pointer, num_tokens < 0, num_seqs <= 0,
 * bad cache), UNSUPPORTED, CUDA; device: BAD_INDEX (seq id, position or block
 * out of range: that token is skipped).  num_tokens == 0 launches nothing.
 */
kvattn_status kvattn_rope_append(const kvattn_config* cfg, const kvattn_cache* cache, void* q,
                                 const void* k, const void* v, const int32_t* positions,
                                 const int32_t* seq_ids, const int32_t* block_table,
                                 int32_t num_seqs, int32_t max_blocks_per_seq, int32_t num_tokens,
                                 void* stream);

/*
 * kvattn_rope_append_strided -- kvattn_rope_append on row-strided q, k, v
 * views, e.g. the three slices of one fused QKV projection output.
 *
 * [Series intro], section 5.1 (and the c_attn row of the weight table in
 * section 5.2): one merged linear layer produces Q, K and V together,
 * [seq_len][3 * hidden], and is then split; with grouped KV heads the row is
 * [Hq*D | Hkv*D | Hkv*D].  Taking the three slices in place avoids copying
 * them out before the rotation:
 *     q = qkv,  k = qkv + Hq*D,  v = qkv + (Hq + Hkv)*D,
 *     q_stride = k_stride = v_stride = (Hq + 2*Hkv)*D.
 *
 *   q_stride    elements from token t's q row to token t+1's (>= Hq*D)
 *   k_stride    the same for k (>= Hkv*D)
 *   v_stride    the same for v (>= Hkv*D)
 *   q_out       device, dense [num_tokens][Hq][D], or NULL: where the rotated
 *               q goes.  NULL rotates q in place (q stays read-write); a
 *               buffer leaves the QKV output as it was and hands the
 *               attention calls a dense q.
 * Inside a row, heads and dimensions are contiguous ([H][D]).  Every row
 * starts on a 16-byte boundary: the base pointers and stride * element size
 * are multiples of 16 bytes.  The rows written (q in place, or q_out) must
 * not overlap any row read by another token or any k or v row.  Everything
 * else, results and errors, as kvattn_rope_append, which is this call with the
 * dense strides Hq*D, Hkv*D, Hkv*D and q_out = NULL.  Errors in addition:
 * INVALID_ARG for a stride below its row length or off the 16-byte rule.
 */
kvattn_status kvattn_rope_append_strided(const kvattn_config* cfg, const kvattn_cache* cache, void* q,
                                         int64_t q_stride, const void* k, int64_t k_stride, const void* v,
                                         int64_t v_stride, void* q_out, const int32_t* positions,
                                         const int32_t* seq_ids, const int32_t* block_table, int32_t num_seqs,
                                         int32_t max_blocks_per_seq, int32_t num_tokens, void* stream);

/*
 * Multi-layer cache: one device allocation holding every layer's K area and V
 * area, so that one block id (one block-table entry, one allocator) names the
 * same block in all of them.
 *
 * [Nano-vLLM], section 05 (5.2): each decoder layer keeps its own K cache
 * area and V cache area, so a logical block index maps to L x 2 physical
 * regions (48 for a 24-layer model), found by arithmetic from the index.
 *
 * Layout of `base`: [num_layers][2 (K, V)][num_blocks][Hkv][block_size][D];
 * layer l's k_pool is region 2l and its v_pool region 2l+1, each a one-layer
 * pool as above.
 *
 * kvattn_layered_cache_bytes: bytes of that allocation (0 for invalid
 * arguments or a size that overflows).
 * kvattn_layer_cache: fills *out with layer `layer`'s one-layer cache (host
 * arithmetic only, nothing launched; base is a device pointer, 16-byte
 * aligned).  Errors: INVALID_ARG (null pointer, layer outside
 * [0, num_layers), num_blocks <= 0, block_size <= 0, misaligned base),
 * UNSUPPORTED (head_dim, group size).
 */
size_t kvattn_layered_cache_bytes(const kvattn_config* cfg, int32_t num_layers, int64_t num_blocks,
                                  int32_t block_size);
kvattn_status kvattn_layer_cache(const kvattn_config* cfg, void* base, int32_t num_layers, int64_t num_blocks,
                                 int32_t block_size, int32_t layer, kvattn_cache* out);

/*
 * kvattn_copy_blocks -- copy-on-write of shared blocks: for i < n, block
 * dst_ids[i] becomes a bit copy of block src_ids[i], in the K and the V pool
 * (kvattn_copy_blocks_layered: in every layer's K and V area of a
 * multi-layer cache, one launch).
 *
 * [Nano-vLLM], section 05: blocks carry reference counts so that sequences
 * with a common prefix share them.  A sequence about to append into a
 * partially filled block that another sequence also references first gets
 * its own copy (kvattn_table_prepare_append names the pair), then appends.
 *
 *   src_ids, dst_ids  device, [n] int32 block ids
 * dst ids must be distinct and none of them a src id of the same call.
 * Errors: INVALID_ARG (null pointer with n > 0, n < 0, bad cache),
 * UNSUPPORTED, CUDA; device: BAD_INDEX (an id outside the pool: that pair is
 * skipped).  n == 0 launches nothing.
 */
kvattn_status kvattn_copy_blocks(const kvattn_config* cfg, const kvattn_cache* cache, const int32_t* src_ids,
                                 const int32_t* dst_ids, int32_t n, void* stream);
kvattn_status kvattn_copy_blocks_layered(const kvattn_config* cfg, void* base, int32_t num_layers,
                                         int64_t num_blocks, int32_t block_size, const int32_t* src_ids,
                                         const int32_t* dst_ids, int32_t n, void* stream);

/*
 * FP8 KV cache: kvattn_rope_append into a kvattn_cache_fp8, and kvattn_decode
 * from it (half the bytes per cached token of bf16, plus 8 bytes of scales
 * per token and KV head).
 *
 * [RoPE page], section 2: besides growing with new tokens and being shared
 * across requests, the KV cache has to support precision compression
 * (16-bit values quantised to 8 bits).  The decode step reads every cached
 * byte, so its time scales with the element size.  e4m3 is taken for the
 * 8-bit format (the GPU converts it to f16 in one instruction per pair).
 *
 * kvattn_rope_append_fp8: as kvattn_rope_append (cfg->dtype must be
 * KVATTN_BF16: q rotated in place in bf16), but each rotated k head row r
 * (its bf16 values, correctly rounded) and each v head row is stored as
 *     amax = max |r|,  scale = amax / 448,  inv = 448 / amax   (fp32, RN;
 *                                                   both 1 when amax = 0)
 *     code = e4m3_rne_satfinite(r * inv)             (the product in fp32, RN)
 * with its scale, in the page layout of kvattn_cache_fp8 (head_dim 128).
 * kvattn_decode_fp8: as kvattn_decode, with K and V the dequantised values
 * code * scale; bf16 q and output, head_dim 128, group size 4 or 8,
 * block_size a multiple of 16 (else UNSUPPORTED / INVALID_ARG).  Workspace:
 * kvattn_decode_workspace_size with the same arguments.
 */
kvattn_status kvattn_rope_append_fp8(const kvattn_config* cfg, const kvattn_cache_fp8* cache, void* q,
                                     const void* k, const void* v, const int32_t* positions, const int32_t* seq_ids,
                                     const int32_t* block_table, int32_t num_seqs, int32_t max_blocks_per_seq,
                                     int32_t num_tokens, void* stream);
kvattn_status kvattn_decode_fp8(const kvattn_config* cfg, const kvattn_cache_fp8* cache, const void* q,
                                const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                int32_t batch, int32_t max_seq_len, int32_t num_splits, void* out, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Workspace bytes kvattn_decode needs for `batch` sequences of at most
 * max_seq_len tokens with num_splits KV splits (0 = the library's choice for
 * the current device; the same arguments give the same choice).
 * Returns 0 for invalid arguments.
 */
size_t kvattn_decode_workspace_size(const kvattn_config* cfg, int32_t batch, int32_t max_seq_len,
                                    int32_t num_splits);

/* The split count kvattn_decode uses for these arguments (num_splits=0 => auto). */
int32_t kvattn_decode_num_splits(const kvattn_config* cfg, int32_t batch, int32_t max_seq_len,
                                 int32_t num_splits);

/*
 * kvattn_decode -- attention of one new query token per sequence against the
 * whole cache of that sequence ([Engine page], section 3.3: with a KV cache
 * the query length is 1 and the mask is (1, S), every cached key visible;
 * section 3.1: softmax(q K^T / sqrt(d_k)) V with d_k = head_dim, scale
 * applied before the softmax).
 *
 *   out[b][j] = sum_{i < seq_lens[b]} softmax_i(q[b][j] . K_b[i][j/G] * scale)
 *               * V_b[i][j/G]
 *
 * The keys of a sequence are split into num_splits ranges processed in
 * parallel, each producing a partial (max, sum, weighted V) that a second
 * kernel merges with the online-softmax rescaling ([Engine page],
 * section 3.4: running max m and running sum l, earlier results rescaled).
 *
 *   q           device, [batch][Hq][D] (already rotated)
 *   block_table device, [batch][max_blocks_per_seq] int32; row b = sequence b
 *   seq_lens    device, [batch] int32, tokens in the cache INCLUDING the new
 *               one (call kvattn_rope_append first); 0 => out row is zeros
 *   max_seq_len host upper bound of seq_lens (a larger length is a BAD_INDEX)
 *   out         device, [batch][Hq][D]
 *   workspace   device, >= kvattn_decode_workspace_size(...) bytes, any
 *               contents, 256-byte aligned; not used after the call returns
 *               except by the work it launched on `stream`.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA; device:
 * BAD_INDEX, TIMEOUT.  batch == 0 launches nothing.
 */
kvattn_status kvattn_decode(const kvattn_config* cfg, const kvattn_cache* cache, const void* q,
                            const int32_t* block_table, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                            int32_t num_splits, void* out, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * kvattn_decode_static_scratch -- kvattn_decode without a caller workspace,
 * for callers that cannot allocate device memory when they run a decode step
 * (for example an engine that has already given nearly all HBM to its own
 * KV-cache pool and arenas, or code inside a host framework's operator
 * interface that has no device allocator and must not call cudaMalloc or
 * cudaFree, which would synchronise the device mid-step).  No counterpart on
 * the pages: it is a deployment convenience of this library.
 *
 * Same arguments, results and errors as kvattn_decode, minus the workspace
 * (the checks of kvattn_decode run first, in its order).  The partial results
 * live in a fixed 32 MiB array in the library's own device memory; a call
 * whose kvattn_decode_workspace_size(cfg, batch, max_seq_len, num_splits)
 * exceeds 32 MiB returns KVATTN_ERR_WORKSPACE_TOO_SMALL and launches nothing.
 * The function allocates nothing itself (no cudaMalloc, cudaFree or
 * allocating library call).
 *
 * Placement: the array is placed on a device (32 MiB of its memory, held
 * until the process exits) by the first call on that device, which also
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current.  Make that first call before sizing your own pools from the free
 * memory, and before any stream capture: the set-up form
 *     kvattn_decode_static_scratch(NULL, NULL, NULL, NULL, 0, NULL, 0, 0, 0, NULL, NULL)
 * (batch 0, cache NULL) does only this and returns KVATTN_OK, or
 * KVATTN_ERR_CUDA if the device has no room for the array (the runtime error
 * is cleared).  Later calls reuse the cached address and need no device
 * memory.  The cached address, like the library's other per-device state,
 * is not valid after cudaDeviceReset on that device.
 *
 * All calls on a device share the one array, so calls whose work overlaps on
 * the GPU (different streams, or concurrent host threads) race and must be
 * serialised by the caller.
 */
kvattn_status kvattn_decode_static_scratch(const kvattn_config* cfg, const kvattn_cache* cache,
                                           const void* q, const int32_t* block_table,
                                           int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                           int32_t batch, int32_t max_seq_len, int32_t num_splits,
                                           void* out, void* stream);

/*
 * kvattn_prefill_chunk -- causal attention of chunks of new query tokens
 * against their sequences' caches, which already hold the chunks' own keys
 * (call kvattn_rope_append for the chunk tokens first).
 * [Series intro], section 2.5 (prefill processes a whole prompt and fills the
 * cache); [Engine page], section 3.3 (each position sees itself and earlier
 * positions) and section 3.4 (tiled attention with an online softmax).
 *
 * Chunk c owns query rows cu_q_lens[c] .. cu_q_lens[c+1]-1 of q; row r of
 * the chunk sits at absolute position prefix_lens[c] + r and sees keys
 * 0 .. prefix_lens[c] + r of block-table row c.
 *
 *   q           device, [total_q][Hq][D] (already rotated), bf16 only
 *   cu_q_lens   device, [num_chunks + 1] int32, cu_q_lens[0] = 0, non-decreasing
 *   prefix_lens device, [num_chunks] int32
 *   block_table device, [num_chunks][max_blocks_per_seq] int32
 *   max_q_len   host upper bound of cu_q_lens[c+1] - cu_q_lens[c]
 *   out         device, [total_q][Hq][D]
 * Uses the tcgen05 tensor cores; needs block_size % 16 == 0 (a contiguous
 * cache then has rows of a multiple of 16 tokens) and head_dim 128 or 64
 * (the GPT-2 shape).  Errors: INVALID_ARG, UNSUPPORTED, CUDA; device:
 * BAD_INDEX, TIMEOUT.  num_chunks == 0 launches nothing.
 */
kvattn_status kvattn_prefill_chunk(const kvattn_config* cfg, const kvattn_cache* cache,
                                   const void* q, const int32_t* cu_q_lens,
                                   const int32_t* prefix_lens, const int32_t* block_table,
                                   int32_t max_blocks_per_seq, int32_t num_chunks,
                                   int32_t max_q_len, int32_t total_q, void* out, void* stream);

/*
 * kvattn_prefill_chunk_fp8 -- kvattn_prefill_chunk over a kvattn_cache_fp8:
 * the same chunks, rows and causal rule, with K and V the dequantised values
 * code * scale rounded to fp32 and then to bf16 (both to nearest even; within
 * half a bf16 ulp plus half an fp32 ulp of code * scale).  [RoPE page],
 * section 2 (the cache compressed to 8 bits); [Engine page], sections 3.3
 * and 3.4.
 *
 * The chunks' pages are first expanded into such a bf16 copy in `workspace`,
 * then the bf16 tensor-core prefill runs over that copy (the compute type of
 * kvattn_prefill_chunk; kvattn_decode_fp8 instead keeps code * scale exact,
 * the codes in f16 and the scales in fp32).
 * cfg->dtype must be KVATTN_BF16 (q and out bf16), head_dim 128, block_size
 * a multiple of 16 (else UNSUPPORTED / INVALID_ARG).
 *
 *   max_kv_tokens  host upper bound of the sum over chunks of
 *                  prefix_lens[c] + (cu_q_lens[c+1] - cu_q_lens[c]); the copy
 *                  holds ceil(max_kv_tokens / block_size) + num_chunks blocks.
 *                  A step whose chunks need more blocks records BAD_INDEX on
 *                  the device and leaves the rows of the chunks past the copy
 *                  unspecified.
 *   workspace      device memory of at least
 *                  kvattn_prefill_fp8_workspace_size(cfg, block_size,
 *                  max_blocks_per_seq, num_chunks, max_kv_tokens) bytes (any
 *                  alignment), owned by the caller, not read before the call
 *                  and free again once the stream has passed it.
 * Other arguments as kvattn_prefill_chunk.  Errors: INVALID_ARG,
 * UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA; device: BAD_INDEX, TIMEOUT.
 * num_chunks == 0 launches nothing.
 */
size_t kvattn_prefill_fp8_workspace_size(const kvattn_config* cfg, int32_t block_size,
                                         int32_t max_blocks_per_seq, int32_t num_chunks,
                                         int64_t max_kv_tokens);
kvattn_status kvattn_prefill_chunk_fp8(const kvattn_config* cfg, const kvattn_cache_fp8* cache,
                                       const void* q, const int32_t* cu_q_lens,
                                       const int32_t* prefix_lens, const int32_t* block_table,
                                       int32_t max_blocks_per_seq, int32_t num_chunks,
                                       int32_t max_q_len, int32_t total_q, int64_t max_kv_tokens,
                                       void* out, void* workspace, size_t workspace_bytes,
                                       void* stream);

/*
 * Waits for `stream`, then returns the device status word of the current
 * device in *out (KVATTN_OK if no kernel recorded an error since the last
 * read) and clears it.  Returns CUDA if the stream itself failed.
 */
kvattn_status kvattn_get_device_status(void* stream, int32_t* out);

/*
 * kvattn_selftest_wait_timeout -- failure-detection self test, no counterpart
 * on the pages.  Launches one CTA that waits on an mbarrier nothing will ever
 * complete, through the same bounded wait every kvattn kernel uses, with a
 * limit of limit_us microseconds (1 .. 1000000).  The wait runs out, the
 * kernel records KVATTN_ERR_TIMEOUT in the device status word and returns; the
 * context stays usable.  INVALID_ARG for a limit out of range.
 */
kvattn_status kvattn_selftest_wait_timeout(int32_t limit_us, void* stream);

/*
 * Host-side block allocator (the CPU "block manager" of [Nano-vLLM],
 * section 05, and the page allocation of [RoPE page], section 5): a free
 * list of fixed-size block ids 0 .. num_blocks-1 in host memory, with a
 * reference count per block (a block shared by several sequences returns to
 * the free list when its last reference is dropped).  Thread-safe.
 */
typedef struct kvattn_allocator kvattn_allocator;

/* INVALID_ARG if num_blocks <= 0 or > 2^31-1 or out == NULL. */
kvattn_status kvattn_allocator_create(int64_t num_blocks, kvattn_allocator** out);
void kvattn_allocator_destroy(kvattn_allocator* a);

/* Takes n free blocks (refcount 1) into out_ids, all or nothing: with fewer
 * than n free it takes none, counts a failure and returns OUT_OF_BLOCKS. */
kvattn_status kvattn_alloc_blocks(kvattn_allocator* a, int32_t n, int32_t* out_ids);

/* Drops one reference of each id; validates all ids first (out of range or
 * not allocated => INVALID_ARG and nothing changes; an id may appear at most
 * as many times as it has references). */
kvattn_status kvattn_free_blocks(kvattn_allocator* a, const int32_t* ids, int32_t n);

/* Takes the given free ids (refcount 1), for adopting an existing block
 * table: INVALID_ARG and nothing changes if one is out of range, not free,
 * or repeated. */
kvattn_status kvattn_claim_blocks(kvattn_allocator* a, const int32_t* ids, int32_t n);

/* Adds one reference to each (allocated) id: INVALID_ARG and nothing changes
 * if one is not allocated. */
kvattn_status kvattn_share_blocks(kvattn_allocator* a, const int32_t* ids, int32_t n);

int64_t kvattn_allocator_num_free(const kvattn_allocator* a);
int64_t kvattn_allocator_num_failures(const kvattn_allocator* a);
int32_t kvattn_allocator_refcount(const kvattn_allocator* a, int32_t id); /* -1 if out of range */

/*
 * Grows one sequence's host block-table row from cur_len to new_len tokens:
 * allocates the blocks for positions cur_len .. new_len-1 that are not yet
 * covered and writes their ids into table_row[cur blocks ...].  All or
 * nothing.  INVALID_ARG if new_len < cur_len or the row is too narrow.
 */
kvattn_status kvattn_table_grow(kvattn_allocator* a, int32_t* table_row, int32_t max_blocks,
                                int32_t block_size, int32_t cur_len, int32_t new_len);

/* Frees the blocks covering a sequence of len tokens and sets those entries to -1. */
kvattn_status kvattn_table_release(kvattn_allocator* a, int32_t* table_row, int32_t max_blocks,
                                   int32_t block_size, int32_t len);

/*
 * Prefix sharing ([Nano-vLLM], section 05: reference-counted blocks shared by
 * sequences with a common prefix).  A new sequence starts as the first len
 * tokens of another: dst_row receives src_row's ids of the blocks covering
 * len tokens and each gains one reference.  All or nothing; INVALID_ARG for a
 * block that is not allocated or a row too narrow.
 */
kvattn_status kvattn_table_fork(kvattn_allocator* a, const int32_t* src_row, int32_t* dst_row,
                                int32_t max_blocks, int32_t block_size, int32_t len);

/*
 * Before appending positions cur_len .. new_len-1 to a sequence: the blocks
 * of kvattn_table_grow, and copy on write of the block that position cur_len
 * falls in when that block is already in the row (cur_len % block_size != 0)
 * and another sequence also references it (refcount > 1).  Then a fresh
 * block replaces it in the row, the old block loses one reference, and
 * *cow_src / *cow_dst name the pair for kvattn_copy_blocks, which must run
 * before the append; otherwise both are -1.  All or nothing: OUT_OF_BLOCKS
 * (one failure counted) leaves the row and every count as they were.
 * INVALID_ARG if new_len < cur_len, the row is too narrow, or the block at
 * cur_len is not allocated.
 */
kvattn_status kvattn_table_prepare_append(kvattn_allocator* a, int32_t* table_row, int32_t max_blocks,
                                          int32_t block_size, int32_t cur_len, int32_t new_len,
                                          int32_t* cow_src, int32_t* cow_dst);

#ifdef __cplusplus
}
#endif
#endif /* KVATTN_H */
