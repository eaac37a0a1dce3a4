// Split-KV decode attention over a paged (or contiguous) KV cache.
//
// What it computes: for every sequence b and query head j,
//   out[b][j] = softmax_i(q[b][j] . K_b[i] * scale) V_b[i],  i < seq_lens[b]
// ("From-scratch AI inference engine" page, section 3.3: with a cache the
// new token's query has length 1 and sees all S cached keys; section 3.1:
// scale 1/sqrt(d_k) before the softmax).  The keys of a sequence are cut into
// chunks; each chunk yields a partial (running max m, running sum l, l-
// normalised weighted V) with the online softmax of section 3.4 of the same
// page, and decode_combine merges the chunks of a sequence.
//
// How (GB300 design):
//  - Persistent grid: every CTA holds a prefix sum of the chunk counts of the
//    batch and walks work items (sequence, chunk, KV head) round-robin, so
//    chunks of equal size spread evenly over the SMs with no empty CTAs.
//  - Warp specialisation: one producer warp streams 16-token tiles of K and V
//    for one KV head (16 x D contiguous elements of one cache block) with
//    1-D TMA bulk copies into an mbarrier-tracked ring of stages; the block
//    ids for 32 upcoming tiles are fetched with one coalesced load.  The ring
//    keeps tens of KB in flight per CTA, which is what HBM needs.
//  - Consumer warps each take whole tiles round-robin and keep their own
//    online-softmax state.  All query heads of a GQA group are computed from
//    the one copy of the tile in shared memory (the KV bytes are read once).
//    A warp splits into token groups; a lane owns a slice of D, computes
//    partial dot products with packed f32x2 FMAs, and a butterfly
//    reduce-scatter over the group's lanes finishes the scores.
//  - All waits are bounded (1 s); on a timeout the CTA records
//    KVATTN_ERR_TIMEOUT and drains without further waiting.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "kvattn_internal.cuh"

namespace kvattn {
namespace {

constexpr int kTile = 16;  // tokens per tile
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxBatch = 8192;  // prefix array lives in shared memory

// --------------------------------------------------------- packed f32x2 math

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

// 16 bytes of cache elements -> f32x2 pairs (element 2i in the low half)
template <bool kBF16>
__device__ __forceinline__ void unpack16(const uint4& w, uint64_t* out)
{
    if constexpr (kBF16) {
        out[0] = pk(bf16lo(w.x), bf16hi(w.x));
        out[1] = pk(bf16lo(w.y), bf16hi(w.y));
        out[2] = pk(bf16lo(w.z), bf16hi(w.z));
        out[3] = pk(bf16lo(w.w), bf16hi(w.w));
    } else {
        out[0] = (uint64_t)w.x | ((uint64_t)w.y << 32);
        out[1] = (uint64_t)w.z | ((uint64_t)w.w << 32);
    }
}

// Butterfly reduce-scatter of N values over the lanes xor-reachable with
// offsets O, O/2, ..., 1: afterwards value i of this lane holds the full sum
// of index (sum over steps of bit*half) + i.
template <int N, int O>
struct Bfly {
    static __device__ __forceinline__ void run(float* v, int lane)
    {
        if constexpr (O >= 1) {
            if constexpr (N > 1) {
                constexpr int H = N / 2;
                const bool up = (lane & O) != 0;
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const float send = up ? v[i] : v[i + H];
                    const float keep = up ? v[i + H] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
                }
                Bfly<H, O / 2>::run(v, lane);
            } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
                Bfly<1, O / 2>::run(v, lane);
            }
        }
    }
};

template <bool kBF16, int kD, int kGT>
struct Traits {
    static constexpr int kE = kBF16 ? 2 : 4;               // bytes per element
    static constexpr int kTG = (kD * kGT > 256) ? 2 : 4;    // token groups per warp
    static constexpr int kLPG = 32 / kTG;                   // lanes per group
    static constexpr int kTPG = kTile / kTG;                // tokens per group per tile
    static constexpr int kDPL = kD / kLPG;                  // dims owned by a lane
    static constexpr int kCE = 16 / kE;                     // elements per 16-byte chunk
    static constexpr int kNC = kDPL / kCE;                  // chunks per lane
    static constexpr int kP = kDPL / 2;                     // f32x2 pairs per lane
    static constexpr int kV = kTPG * kGT;                   // partial scores per lane
    static constexpr int kR = kV >= kLPG ? kV / kLPG : 1;   // scores per lane after reduction
    static constexpr int kBW = kV >= kLPG ? kTPG / kR : kLPG;  // lanes sharing one head's scores
    static constexpr int kDup = kV >= kLPG ? 1 : kLPG / kV;    // lanes holding the same score
    static constexpr int kTileBytes = kTile * kD * kE;      // K (or V) bytes of a full tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static_assert(kNC >= 1 && kDPL % kCE == 0, "lane slice must hold whole 16-byte chunks");
    static_assert(kBW >= 1, "head block");
};

struct SharedLayout {
    int stages;
    int ring_off, merge_off, pbuf_off, prefix_off, bar_off, flag_off, bytes;
};

template <bool kBF16, int kD, int kGT>
__host__ __device__ inline SharedLayout shared_layout(int stages, int batch)
{
    using T = Traits<kBF16, kD, kGT>;
    SharedLayout L;
    L.stages = stages;
    int off = 0;
    L.ring_off = off;
    off += stages * T::kStageBytes;
    L.merge_off = off;
    off += kConsumerWarps * kGT * (kD + 2) * 4;
    L.pbuf_off = off;
    off += kConsumerWarps * T::kTG * T::kV * 4;
    L.prefix_off = off;
    off += ((batch + 1) * 4 + 15) / 16 * 16;
    L.bar_off = off;
    off += 2 * stages * 8;
    L.flag_off = off;
    off += 16;
    L.bytes = off;
    return L;
}

struct ItemInfo {
    int b, chunk, h, hsub, nchunks, len;
};

// Work item `idx` -> (sequence, chunk, kv head, q-head subgroup) and its tiles.
__device__ __forceinline__ ItemInfo decode_item(int idx, const int* prefix, int batch, int heads_x_sub,
                                                int nsub, const DecodeArgs& a)
{
    ItemInfo it;
    const int hh = idx % heads_x_sub;
    const int rest = idx / heads_x_sub;
    // first b with prefix[b+1] > rest
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid + 1] > rest) hi = mid; else lo = mid + 1;
    }
    it.b = lo;
    it.chunk = rest - prefix[lo];
    it.nchunks = prefix[lo + 1] - prefix[lo];
    it.h = hh / nsub;
    it.hsub = hh - it.h * nsub;
    int L = a.seq_lens[it.b];
    if (L < 0 || L > a.max_seq_len || (int64_t)L > (int64_t)a.max_blocks * a.block_size) L = 0;
    it.len = L;
    return it;
}

template <bool kBF16, int kD, int kGT>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const __grid_constant__ DecodeArgs a,
                                                                const int stages)
{
    const int chunk_tiles = a.chunk_tiles;
    using T = Traits<kBF16, kD, kGT>;
    extern __shared__ __align__(1024) unsigned char smem[];
    const SharedLayout SL = shared_layout<kBF16, kD, kGT>(stages, a.batch);
    unsigned char* ring = smem + SL.ring_off;
    float* merge = reinterpret_cast<float*>(smem + SL.merge_off);
    float* pbuf_all = reinterpret_cast<float*>(smem + SL.pbuf_off);
    int* prefix = reinterpret_cast<int*>(smem + SL.prefix_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SL.bar_off);
    uint64_t* empty = full + stages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL.flag_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.hq / a.hkv;
    const int nsub = G / kGT;
    const int heads_x_sub = a.hkv * nsub;

    // ---- per-sequence chunk counts and their exclusive prefix sum
    for (int b = tid; b < a.batch; b += kThreads) {
        int L = a.seq_lens[b];
        if (L < 0 || L > a.max_seq_len || (int64_t)L > (int64_t)a.max_blocks * a.block_size) {
            record_error(a.status, KVATTN_ERR_BAD_INDEX);
            L = 0;
        }
        const int nt = (L + kTile - 1) / kTile;
        prefix[b + 1] = max(1, (nt + chunk_tiles - 1) / chunk_tiles);
    }
    if (tid == 0) {
        prefix[0] = 0;
        *abort_flag = 0;
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {  // inclusive scan of prefix[1..batch] by one warp
        const int per = (a.batch + 31) / 32;
        const int beg = 1 + lane * per, end = min(a.batch + 1, beg + per);
        int s = 0;
        for (int i = beg; i < end; ++i) s += prefix[i];
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int run = incl - s;
        for (int i = beg; i < end; ++i) {
            run += prefix[i];
            prefix[i] = run;
        }
    }
    __syncthreads();
    const int num_items = prefix[a.batch] * heads_x_sub;

    if (warp == kConsumerWarps) {
        // =========================== producer warp ===========================
        const uint64_t policy = l2_evict_first_policy();
        uint32_t pos = 0;  // stream position (tiles issued by this CTA)
        for (int idx = blockIdx.x; idx < num_items; idx += gridDim.x) {
            ItemInfo it = decode_item(idx, prefix, a.batch, heads_x_sub, nsub, a);
            const int nt = (it.len + kTile - 1) / kTile;
            const int t0 = it.chunk * chunk_tiles;
            const int t1 = min(nt, t0 + chunk_tiles);
            for (int base = t0; base < t1; base += 32) {
                // block ids of the next 32 tiles, one coalesced load
                const int ti = base + lane;
                int64_t blk = 0;
                bool ok = true;
                if (ti < t1) {
                    const int tok = ti * kTile;
                    const int32_t v = a.block_table[(int64_t)it.b * a.max_blocks + tok / a.block_size];
                    ok = v >= 0 && v < a.num_blocks;
                    blk = ok ? v : 0;
                }
                if (!ok) record_error(a.status, KVATTN_ERR_BAD_INDEX);
                const int cnt = min(32, t1 - base);
                for (int j = 0; j < cnt; ++j) {
                    const int64_t bj = __shfl_sync(0xffffffffu, blk, j);
                    if (lane == 0) {
                        const uint32_t stage = pos % stages, use = pos / stages;
                        bool go = !*abort_flag;
                        if (go && use > 0) go = mbar_wait(&empty[stage], (use - 1) & 1, a.status);
                        if (!go) {
                            *abort_flag = 1;
                        } else {
                            const int tok = (base + j) * kTile;
                            const int nvalid = min(kTile, it.len - tok);
                            const uint32_t bytes = (uint32_t)nvalid * kD * T::kE;
                            const int64_t row = (bj * a.hkv + it.h) * a.block_size + tok % a.block_size;
                            const char* ksrc = (const char*)a.k_pool + row * kD * T::kE;
                            const char* vsrc = (const char*)a.v_pool + row * kD * T::kE;
                            unsigned char* dst = ring + (size_t)stage * T::kStageBytes;
                            mbar_arrive_expect_tx(&full[stage], 2 * bytes);
                            bulk_load(dst, ksrc, bytes, &full[stage], policy);
                            bulk_load(dst + T::kTileBytes, vsrc, bytes, &full[stage], policy);
                        }
                    }
                    ++pos;
                }
            }
        }
        // drain: every issued copy must land before the CTA exits
        if (lane == 0 && *abort_flag) {
            const uint32_t n = pos < (uint32_t)stages ? pos : (uint32_t)stages;
            for (uint32_t p = pos - n; p < pos; ++p) mbar_wait(&full[p % stages], (p / stages) & 1, a.status);
        }
        return;
    }

    // ============================== consumer warps ==============================
    const int grp = lane / T::kLPG;      // token group inside the warp
    const int sub = lane % T::kLPG;      // lane inside the group
    float* pbuf = pbuf_all + warp * T::kTG * T::kV + grp * T::kV;
    const int hq = a.hq;
    uint32_t pos = 0;

    for (int idx = blockIdx.x; idx < num_items; idx += gridDim.x) {
        ItemInfo it = decode_item(idx, prefix, a.batch, heads_x_sub, nsub, a);
        const int nt = (it.len + kTile - 1) / kTile;
        const int t0 = it.chunk * chunk_tiles;
        const int t1 = min(nt, t0 + chunk_tiles);
        const int ntiles = max(0, t1 - t0);
        const int qh0 = it.h * G + it.hsub * kGT;  // first query head of this item

        // query slice of this lane, pre-scaled by scale*log2(e)
        uint64_t q2[kGT][T::kP];
#pragma unroll
        for (int g = 0; g < kGT; ++g) {
            const char* qrow = (const char*)a.q + ((int64_t)it.b * hq + qh0 + g) * kD * T::kE;
#pragma unroll
            for (int c = 0; c < T::kNC; ++c) {
                const int e0 = c * T::kLPG * T::kCE + sub * T::kCE;
                const uint4 w = *reinterpret_cast<const uint4*>(qrow + e0 * T::kE);
                uint64_t tmp[4];
                unpack16<kBF16>(w, tmp);
#pragma unroll
                for (int i = 0; i < T::kCE / 2; ++i)
                    q2[g][c * (T::kCE / 2) + i] = fmul2(tmp[i], pk(a.scale_log2, a.scale_log2));
            }
        }
        uint64_t acc[kGT][T::kP];
        float m[kGT], lsum[kGT];
#pragma unroll
        for (int g = 0; g < kGT; ++g) {
            m[g] = -INFINITY;
            lsum[g] = 0.f;
#pragma unroll
            for (int i = 0; i < T::kP; ++i) acc[g][i] = 0;
        }

        for (int li = 0; li < ntiles; ++li) {
            const uint32_t p = pos + li;
            if ((int)(p % kConsumerWarps) != warp) continue;
            const uint32_t stage = p % stages;
            bool ready = !*abort_flag;
            if (ready) ready = mbar_wait(&full[stage], (p / stages) & 1, a.status);
            ready = __all_sync(0xffffffffu, ready);
            if (!ready) {
                if (lane == 0) *abort_flag = 1;
                continue;
            }
            const unsigned char* ks = ring + (size_t)stage * T::kStageBytes;
            const unsigned char* vs = ks + T::kTileBytes;
            const int tok0 = (t0 + li) * kTile;
            const int nvalid = min(kTile, it.len - tok0);

            // ---- partial scores of this lane's tokens and heads
            float sc[T::kV];
#pragma unroll
            for (int t = 0; t < T::kTPG; ++t) {
                const int row = grp * T::kTPG + t;
                uint64_t k2[T::kP];
#pragma unroll
                for (int c = 0; c < T::kNC; ++c) {
                    const int e0 = c * T::kLPG * T::kCE + sub * T::kCE;
                    const uint4 w = *reinterpret_cast<const uint4*>(ks + (row * kD + e0) * T::kE);
                    unpack16<kBF16>(w, &k2[c * (T::kCE / 2)]);
                }
#pragma unroll
                for (int g = 0; g < kGT; ++g) {
                    uint64_t s2 = ffma2(q2[g][0], k2[0], 0ull);
#pragma unroll
                    for (int i = 1; i < T::kP; ++i) s2 = ffma2(q2[g][i], k2[i], s2);
                    sc[g * T::kTPG + t] = pk_lo(s2) + pk_hi(s2);
                }
            }
            Bfly<T::kV, T::kLPG / 2>::run(sc, lane);

            // ---- scores held by this lane: mask, group max per head
            float bmax = -INFINITY;  // max of this lane's scores (all belong to one head)
            int my_g;
#pragma unroll
            for (int r = 0; r < T::kR; ++r) {
                const int idxv = T::kV >= T::kLPG ? sub * T::kR + r : sub / T::kDup;
                const int tt = idxv % T::kTPG;
                my_g = idxv / T::kTPG;
                if (grp * T::kTPG + tt >= nvalid) sc[r] = -INFINITY;
                bmax = fmaxf(bmax, sc[r]);
            }
#pragma unroll
            for (int o = T::kBW / 2; o >= 1; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
            // every lane of the group learns the tile max of every head
            float mnew[kGT], alpha[kGT];
            bool grow = false;
#pragma unroll
            for (int g = 0; g < kGT; ++g) {
                const float tm = __shfl_sync(0xffffffffu, bmax, grp * T::kLPG + g * T::kBW);
                mnew[g] = fmaxf(m[g], tm);
                alpha[g] = (mnew[g] == -INFINITY) ? 1.f : exp2f(m[g] - mnew[g]);
                grow |= mnew[g] != m[g];
            }
            // probabilities of this lane's scores
            float mine_m = mnew[0];
#pragma unroll
            for (int g = 1; g < kGT; ++g)
                if (my_g == g) mine_m = mnew[g];
            float lpart = 0.f;
#pragma unroll
            for (int r = 0; r < T::kR; ++r) {
                const float pv = (sc[r] == -INFINITY) ? 0.f : exp2f(sc[r] - mine_m);
                sc[r] = pv;
                lpart += pv;
            }
            if (T::kDup > 1 && (sub % T::kDup) != 0) lpart = 0.f;
#pragma unroll
            for (int g = 0; g < kGT; ++g) {
                lsum[g] = lsum[g] * alpha[g] + (my_g == g ? lpart : 0.f);
                m[g] = mnew[g];
            }
            if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int g = 0; g < kGT; ++g) {
                    const uint64_t a2 = pk(alpha[g], alpha[g]);
#pragma unroll
                    for (int i = 0; i < T::kP; ++i) acc[g][i] = fmul2(acc[g][i], a2);
                }
            }
            // ---- share probabilities inside the group
#pragma unroll
            for (int r = 0; r < T::kR; ++r) {
                const int idxv = T::kV >= T::kLPG ? sub * T::kR + r : sub / T::kDup;
                pbuf[idxv] = sc[r];
            }
            __syncwarp();
            // ---- weighted V
#pragma unroll
            for (int t = 0; t < T::kTPG; ++t) {
                const int row = grp * T::kTPG + t;
                if (row < nvalid) {
                    uint64_t v2[T::kP];
#pragma unroll
                    for (int c = 0; c < T::kNC; ++c) {
                        const int e0 = c * T::kLPG * T::kCE + sub * T::kCE;
                        const uint4 w = *reinterpret_cast<const uint4*>(vs + (row * kD + e0) * T::kE);
                        unpack16<kBF16>(w, &v2[c * (T::kCE / 2)]);
                    }
#pragma unroll
                    for (int g = 0; g < kGT; ++g) {
                        const float pw = pbuf[g * T::kTPG + t];
                        const uint64_t p2 = pk(pw, pw);
#pragma unroll
                        for (int i = 0; i < T::kP; ++i) acc[g][i] = ffma2(p2, v2[i], acc[g][i]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
        }
        pos += ntiles;

        // ---- merge the token groups of this warp
#pragma unroll
        for (int g = 0; g < kGT; ++g) {
            float l = lsum[g];
#pragma unroll
            for (int o = T::kLPG / 2; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            float M = m[g];
#pragma unroll
            for (int o = T::kLPG; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float f = (m[g] == -INFINITY) ? 0.f : exp2f(m[g] - M);
            l *= f;
            const uint64_t f2 = pk(f, f);
#pragma unroll
            for (int i = 0; i < T::kP; ++i) acc[g][i] = fmul2(acc[g][i], f2);
#pragma unroll
            for (int o = T::kLPG; o < 32; o <<= 1) {
                l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
                for (int i = 0; i < T::kP; ++i) {
                    const uint64_t other = __shfl_xor_sync(0xffffffffu, acc[g][i], o);
                    acc[g][i] = pk(pk_lo(acc[g][i]) + pk_lo(other), pk_hi(acc[g][i]) + pk_hi(other));
                }
            }
            m[g] = M;
            lsum[g] = l;
        }
        // ---- write this warp's state, merge the warps
        float* mw = merge + (size_t)warp * kGT * (kD + 2);
        if (grp == 0) {
#pragma unroll
            for (int g = 0; g < kGT; ++g) {
#pragma unroll
                for (int c = 0; c < T::kNC; ++c) {
#pragma unroll
                    for (int i = 0; i < T::kCE / 2; ++i) {
                        const int e = c * T::kLPG * T::kCE + sub * T::kCE + 2 * i;
                        const uint64_t v = acc[g][c * (T::kCE / 2) + i];
                        mw[g * (kD + 2) + e] = pk_lo(v);
                        mw[g * (kD + 2) + e + 1] = pk_hi(v);
                    }
                }
                if (sub == 0) {
                    mw[g * (kD + 2) + kD] = m[g];
                    mw[g * (kD + 2) + kD + 1] = lsum[g];
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
        const bool direct = it.nchunks == 1;
        for (int e = tid; e < kGT * kD; e += kConsumerWarps * 32) {
            const int g = e / kD, d = e - g * kD;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, merge[(w * kGT + g) * (kD + 2) + kD]);
            float num = 0.f, den = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float* mr = merge + (size_t)(w * kGT + g) * (kD + 2);
                    const float f = (mr[kD] == -INFINITY) ? 0.f : exp2f(mr[kD] - M);
                    num += f * mr[d];
                    den += f * mr[kD + 1];
                }
            }
            const float o = den > 0.f ? num / den : 0.f;
            const int64_t qrow = (int64_t)it.b * hq + qh0 + g;
            if (direct) {
                if constexpr (kBF16)
                    reinterpret_cast<__nv_bfloat16*>(a.out)[qrow * kD + d] = __float2bfloat16_rn(o);
                else
                    reinterpret_cast<float*>(a.out)[qrow * kD + d] = o;
            } else {
                const int64_t prow = qrow * a.splits + it.chunk;
                a.part_o[prow * kD + d] = o;
                if (d == 0) {
                    a.part_ml[prow * 2] = M;
                    a.part_ml[prow * 2 + 1] = den;
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    }
}

// Merge the chunk partials of the sequences that have more than one chunk.
template <bool kBF16, int kD>
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__ DecodeArgs a)
{
    const int chunk_tiles = a.chunk_tiles;
    const int wid = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (wid >= a.batch * a.hq) return;
    const int b = wid / a.hq;
    int L = a.seq_lens[b];
    if (L < 0 || L > a.max_seq_len || (int64_t)L > (int64_t)a.max_blocks * a.block_size) L = 0;
    const int nt = (L + kTile - 1) / kTile;
    const int nc = max(1, (nt + chunk_tiles - 1) / chunk_tiles);
    if (nc == 1) return;
    constexpr int kDL = kD / 32;
    const float* ml = a.part_ml + (int64_t)wid * a.splits * 2;
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, ml[2 * c]);
    float acc[kDL];
#pragma unroll
    for (int i = 0; i < kDL; ++i) acc[i] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
        for (int c = 0; c < nc; ++c) {
            const float mc = ml[2 * c], lc = ml[2 * c + 1];
            const float w = (mc == -INFINITY) ? 0.f : lc * exp2f(mc - M);
            den += w;
            const float* o = a.part_o + ((int64_t)wid * a.splits + c) * kD;
#pragma unroll
            for (int i = 0; i < kDL; ++i) acc[i] += w * o[lane * kDL + i];
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int i = 0; i < kDL; ++i) {
        const int64_t e = (int64_t)wid * kD + lane * kDL + i;
        if constexpr (kBF16)
            reinterpret_cast<__nv_bfloat16*>(a.out)[e] = __float2bfloat16_rn(acc[i] * inv);
        else
            reinterpret_cast<float*>(a.out)[e] = acc[i] * inv;
    }
}

struct LaunchCfg {
    int stages = 0, ctas_per_sm = 0, smem = 0;
};

template <bool kBF16, int kD, int kGT>
kvattn_status run(const DecodeArgs& a, cudaStream_t s)
{
    const int chunk_tiles = a.chunk_tiles;
    using T = Traits<kBF16, kD, kGT>;
    // ring depth: about 64 KB of stages per CTA
    const int stages = std::max(4, std::min(16, 65536 / T::kStageBytes));
    const SharedLayout SL = shared_layout<kBF16, kD, kGT>(stages, a.batch);
    auto kern = decode_split_kernel<kBF16, kD, kGT>;
    static std::mutex mu;
    static int configured_smem = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        if (SL.bytes > configured_smem) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SL.bytes);
            if (e != cudaSuccess) return KVATTN_ERR_CUDA;
            configured_smem = SL.bytes;
        }
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, SL.bytes) != cudaSuccess)
        return KVATTN_ERR_CUDA;
    per_sm = std::max(1, per_sm);
    const int G = a.hq / a.hkv;
    int64_t items_upper = 0;
    {
        const int max_tiles = (a.max_seq_len + kTile - 1) / kTile;
        const int max_chunks = std::max(1, (max_tiles + chunk_tiles - 1) / chunk_tiles);
        items_upper = (int64_t)a.batch * max_chunks * a.hkv * (G / kGT);
    }
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(items_upper, (int64_t)num_sms() * per_sm));
    kern<<<(unsigned)grid, kThreads, SL.bytes, s>>>(a, stages);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return KVATTN_ERR_CUDA;
    if (a.splits > 1) {
        const int warps = a.batch * a.hq;
        decode_combine_kernel<kBF16, kD><<<(warps + 3) / 4, 128, 0, s>>>(a);
        e = cudaGetLastError();
    }
    return cuda_status(e);
}

}  // namespace

DecodePlan decode_plan(int32_t batch, int32_t hkv, int32_t group, int32_t max_seq_len, int32_t splits)
{
    const int max_tiles = std::max(1, (max_seq_len + kTile - 1) / kTile);
    int chunk;
    if (splits > 0) {
        chunk = (max_tiles + splits - 1) / splits;
    } else {
        // Enough equal-sized chunks for every CTA slot to receive ~16 of them
        // (static round-robin then balances to a few percent), but at least 8
        // tiles per chunk so the fixed cost of a chunk stays small.
        const int nsub = group > 4 ? group / 4 : 1;
        const int64_t slots = (int64_t)num_sms() * 2;
        const int64_t pairs = (int64_t)batch * hkv * nsub;
        const double avg_tiles = std::max(1.0, max_tiles * 0.5);
        chunk = (int)std::floor(pairs * avg_tiles / (16.0 * slots));
        chunk = std::max(8, std::min(chunk, max_tiles));
    }
    DecodePlan p;
    p.chunk_tiles = std::max(1, chunk);
    p.max_chunks = (max_tiles + p.chunk_tiles - 1) / p.chunk_tiles;
    return p;
}

kvattn_status launch_decode(const DecodeArgs& a, cudaStream_t s)
{
    const int G = a.hq / a.hkv;
    const bool bf16 = a.dtype == KVATTN_BF16;
    const int gt = G >= 4 ? 4 : G;
#define KVATTN_DECODE_CASE(BF, DD, GG) \
    if (bf16 == BF && a.d == DD && gt == GG) return run<BF, DD, GG>(a, s);
    KVATTN_DECODE_CASE(true, 128, 1)
    KVATTN_DECODE_CASE(true, 128, 2)
    KVATTN_DECODE_CASE(true, 128, 4)
    KVATTN_DECODE_CASE(true, 64, 1)
    KVATTN_DECODE_CASE(true, 64, 2)
    KVATTN_DECODE_CASE(true, 64, 4)
    KVATTN_DECODE_CASE(false, 128, 1)
    KVATTN_DECODE_CASE(false, 128, 2)
    KVATTN_DECODE_CASE(false, 128, 4)
    KVATTN_DECODE_CASE(false, 64, 1)
    KVATTN_DECODE_CASE(false, 64, 2)
    KVATTN_DECODE_CASE(false, 64, 4)
#undef KVATTN_DECODE_CASE
    return KVATTN_ERR_UNSUPPORTED;
}

}  // namespace kvattn
