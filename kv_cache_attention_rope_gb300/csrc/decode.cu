// Split-KV decode attention over a paged (or contiguous) KV cache.
//
// What it computes: for every sequence b and query head j,
//   out[b][j] = softmax_i(q[b][j] . K_b[i] * scale) V_b[i],  i < seq_lens[b]
// ("From-scratch AI inference engine" page, section 3.3: with a cache the
// new token's query has length 1 and sees all S cached keys; section 3.1:
// scale 1/sqrt(d_k) before the softmax).  The keys of a sequence may be cut
// into pieces; each piece yields a partial (running max m, running sum l,
// l-normalised weighted V) with the online softmax of section 3.4 of the same
// page, and decode_combine merges the pieces of a sequence.
//
// How (GB300 design):
//  - Flat work decomposition: the 16-token tiles of all (sequence, KV head)
//    segments form one stream; every persistent CTA takes an equal
//    contiguous range of it (segments are cut where ranges meet), so the
//    load is balanced to one tile whatever the length mix.  Each CTA derives
//    the ranges from a prefix sum of the batch's tile counts held in shared
//    memory.  A cap on the pieces per segment bounds the workspace.
//  - Warp specialisation: one producer warp streams tiles of K and V (16 x D
//    contiguous elements of one block and KV head) with 1-D TMA bulk copies
//    into an mbarrier-tracked ring of stages; the block ids of the next 32
//    tiles come from one coalesced load.  The ring keeps tens of KB in flight
//    per CTA, which is what HBM needs.
//  - Consumer warps take whole tiles round-robin and keep their own
//    online-softmax state.  All query heads of a GQA group are computed from
//    the one copy of a tile in shared memory (KV bytes are read once).  A warp
//    splits into token groups; a lane owns a slice of D, forms partial dot
//    products with packed f32x2 FMAs, and a select-free butterfly
//    reduce-scatter over the group's lanes finishes the scores (each lane
//    holds its partials in a lane-dependent XOR order so that every level
//    keeps the lower half and receives the upper half).
//  - All waits are bounded (1 s); on a timeout the CTA records
//    KVATTN_ERR_TIMEOUT and drains without further waiting.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "kvattn_tc.cuh"

namespace kvattn {
namespace {

constexpr int kTile = 16;  // tokens per tile
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMinPer = 4;  // fewest tiles in a CTA's range (flat mode)
// residency the register and shared-memory budgets aim at: 3 CTAs per SM
// (the tensor-core path keeps only rows 0..7 of its 16 x 8 fragments, which
// fits it in 128 registers; at 3 CTAs it reads c4 at the HBM copy rate, at 2
// CTAs with more registers it reached 90%).  The fp8 path runs 4 CTAs
// (96 registers): its 4 KB pages need more producers issuing copies and more
// consumer warps hiding MMA latency per byte than the 8 KB bf16 tiles.
template <bool kMma, bool kFP8 = false>
constexpr int ctas_per_sm() { return kFP8 ? 4 : 3; }

// Tensor maps of the K and V pools (tensor-core path).  Blocks of a multiple
// of 16 tokens: one 4-D box per 16-token page, stage layout [8-row group]
// [64-column panel][8 rows][128 B].  Otherwise (a contiguous cache of any
// length): two 2-D boxes per page from any first row, layout [64-column
// panel][16 rows][128 B].  The consumer only swaps two strides.
struct PageMaps {
    CUtensorMap k, v;
};

// 2^x (ex2.approx.ftz: a few ulp, far below the bf16 rounding P goes through
// on the tensor-core path); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

// Select-free butterfly reduce-scatter of N values over lanes xor-reachable
// with offsets O, O/2, ..., 1.  Every level keeps the lower half and adds the
// partner's upper half; that is a reduce-scatter because each lane stores its
// values XOR-permuted by a lane-dependent mask (see Traits::mask).
template <int N, int O>
struct Bfly {
    static __device__ __forceinline__ void run(float* v)
    {
        if constexpr (O >= 1) {
            if constexpr (N > 1) {
                constexpr int H = N / 2;
#pragma unroll
                for (int i = 0; i < H; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + H], O);
                Bfly<H, O / 2>::run(v);
            } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
                Bfly<1, O / 2>::run(v);
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
    static_assert(kBW >= 1 && kTPG % 2 == 0, "tile split");
    // logical score index held first by this lane after the reduction; it is
    // also the XOR mask of the lane's partial-score layout
    static __device__ __forceinline__ int mask(int sub) { return kV >= kLPG ? sub * kR : sub / kDup; }
};

struct SharedLayout {
    int ring_off, merge_off, pbuf_off, prefix_off, bar_off, flag_off, bytes;  // pbuf aliases merge
};

// Bytes of one ring stage: K and V pages of a tile (one fp8 page for an fp8 cache).
template <bool kBF16, int kD, int kGT, bool kFP8>
__host__ __device__ constexpr int stage_bytes() { return kFP8 ? kF8Page : Traits<kBF16, kD, kGT>::kStageBytes; }

// Query heads a consumer warp merges per pass (its merge slot's size): a
// GQA group of 8 on the tensor cores is merged in two passes of 4, which keeps
// the slot, and with it the ring depth, as for groups of 4.  The fp8 path
// merges one head per pass: its 4 KB pages leave room for 12 ring stages at 4
// CTAs per SM only with the smaller slot (8 stages with slots of 4 heads).
template <int kGT, bool kFP8 = false>
__host__ __device__ constexpr int merge_heads() { return kFP8 ? 1 : kGT < 4 ? kGT : 4; }

template <bool kBF16, int kD, int kGT, bool kFP8 = false>
__host__ __device__ inline SharedLayout shared_layout(int stages, int batch)
{
    using T = Traits<kBF16, kD, kGT>;
    SharedLayout L;
    int off = 0;
    L.ring_off = off;
    off += stages * stage_bytes<kBF16, kD, kGT, kFP8>();
    // per consumer warp: its merge slot (kGT x (D + 2) floats, written at the
    // end of a piece) doubles as its probability buffer while tiles stream
    constexpr int kMG = merge_heads<kGT, kFP8>();
    static_assert(kMG == kGT || kGT > 4 || kFP8, "only groups above 4 and fp8 pages are merged in passes");
    static_assert(kGT > 4 || kFP8 || T::kTG * T::kV * 8 <= kMG * (kD + 2) * 4,
                  "probability buffer fits the merge slot");
    L.merge_off = off;
    off += kConsumerWarps * kMG * (kD + 2) * 4;
    L.pbuf_off = L.merge_off;
    L.prefix_off = off;
    off += ((batch + 1) * 4 + 15) / 16 * 16;
    L.bar_off = off;
    off += 2 * stages * 8;
    L.flag_off = off;
    off += 16;
    L.bytes = off;
    return L;
}

// One contiguous run of tiles of one (sequence, KV head [, q-head subgroup])
// segment, and where its result goes.
struct Piece {
    int b, hh, t0, t1, len;
    int slot, nslots;  // partial slot of this piece among the segment's pieces
};

// Walks the pieces of this CTA.  Producer and consumers run identical copies.
struct PieceIter {
    const int* P;  // P[b]: first stream tile of sequence b (P[batch] = total)
    int batch, hh_count, per, r, r1, b, seg;
    bool flat;

    __device__ bool next(Piece& pc, const DecodeArgs& a)
    {
        if (flat) {
            if (r >= r1) return false;
            while (P[b + 1] <= r) ++b;
            const int nt = (P[b + 1] - P[b]) / hh_count;
            const int off = r - P[b];
            const int hh = off / nt;
            const int t0 = off - hh * nt;
            const int take = min(nt - t0, r1 - r);
            const int s0 = P[b] + hh * nt;
            const int first = s0 / per, last = (s0 + nt - 1) / per;
            pc.b = b;
            pc.hh = hh;
            pc.t0 = t0;
            pc.t1 = t0 + take;
            pc.slot = (int)blockIdx.x - first;
            pc.nslots = last - first + 1;
            r += take;
        } else {
            while (true) {
                if (seg >= batch * hh_count) return false;
                const int bb = seg / hh_count, hh = seg - bb * hh_count;
                const int nt = (P[bb + 1] - P[bb]) / hh_count;
                seg += gridDim.x;
                if (nt == 0) continue;
                pc.b = bb;
                pc.hh = hh;
                pc.t0 = 0;
                pc.t1 = nt;
                pc.slot = 0;
                pc.nslots = 1;
                break;
            }
        }
        pc.len = a.seq_lens[pc.b];
        return true;
    }
};

__device__ __forceinline__ bool len_ok(int L, const DecodeArgs& a)
{
    return L >= 0 && L <= a.max_seq_len && (int64_t)L <= (int64_t)a.max_blocks * a.block_size;
}

template <bool kBF16, int kD, int kGT, bool kMma, bool kRowBoxes, bool kFP8 = false>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<kMma, kFP8>()) decode_split_kernel(const __grid_constant__ DecodeArgs a,
                                                                const __grid_constant__ PageMaps maps,
                                                                const int stages)
{
    pdl_wait();
    using T = Traits<kBF16, kD, kGT>;
    static_assert(!kMma || (kBF16 && kD == 128 && kGT <= 8), "tensor-core path: bf16, D = 128, <= 8 heads");
    static_assert(!kFP8 || (kMma && !kRowBoxes), "fp8 cache: tensor-core path on 16-row pages");
    constexpr int kStageB = stage_bytes<kBF16, kD, kGT, kFP8>();
    extern __shared__ unsigned char smem_raw[];
    // 1 KB alignment: the tensor-core path's stages hold 128-byte-swizzled pages
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const SharedLayout SL = shared_layout<kBF16, kD, kGT, kFP8>(stages, a.batch);
    unsigned char* ring = smem + SL.ring_off;
    float* merge = reinterpret_cast<float*>(smem + SL.merge_off);
    int* prefix = reinterpret_cast<int*>(smem + SL.prefix_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SL.bar_off);
    uint64_t* empty = full + stages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL.flag_off);
    int* max_nt_sh = reinterpret_cast<int*>(smem + SL.flag_off + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.hq / a.hkv;
    const int nsub = G / kGT;
    const int HH = a.hkv * nsub;  // segments per sequence

    // ---- tiles per segment of each sequence, prefix sum over the batch
    for (int b = tid; b < a.batch; b += kThreads) {
        const int L = a.seq_lens[b];
        int nt = 0;
        if (len_ok(L, a)) nt = (L + kTile - 1) / kTile;
        else if (blockIdx.x == 0) record_error(a.status, KVATTN_ERR_BAD_INDEX);
        prefix[b + 1] = nt;
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
    if (warp == 0) {  // prefix[i] <- HH * (tiles of sequences 0..i-1); max tiles of one sequence
        const int per = (a.batch + 31) / 32;
        const int beg = 1 + lane * per, end = min(a.batch + 1, beg + per);
        int s = 0, mx = 0;
        for (int i = beg; i < end; ++i) {
            s += prefix[i];
            mx = max(mx, prefix[i]);
        }
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        int run = incl - s;
        for (int i = beg; i < end; ++i) {
            run += prefix[i];
            prefix[i] = run * HH;
        }
        if (lane == 0) *max_nt_sh = mx;
    }
    __syncthreads();

    // ---- sequences with no keys (or an invalid length): zero output
    for (int b = blockIdx.x; b < a.batch; b += gridDim.x) {
        if (prefix[b + 1] != prefix[b]) continue;
        for (int e = tid; e < a.hq * kD; e += kThreads) {
            const int64_t o = (int64_t)b * a.hq * kD + e;
            if constexpr (kBF16) reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(0.f);
            else reinterpret_cast<float*>(a.out)[o] = 0.f;
        }
        if (a.nslots)
            for (int h = tid; h < HH; h += kThreads) a.nslots[(int64_t)b * HH + h] = 1;
    }

    PieceIter iter;
    iter.P = prefix;
    iter.batch = a.batch;
    iter.hh_count = HH;
    iter.b = 0;
    iter.flat = a.splits > 1;
    {
        const int total = prefix[a.batch];
        const int max_nt = *max_nt_sh;
        int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
        if (iter.flat) per = max(per, (max_nt + a.splits - 2) / (a.splits - 1));
        per = max(per, kMinPer);
        iter.per = per;
        iter.r = min(total, (int)blockIdx.x * per);
        iter.r1 = min(total, iter.r + per);
        if (iter.flat && iter.r < iter.r1) {  // first sequence of the range
            int lo = 0, hi = a.batch - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (prefix[mid + 1] > iter.r) hi = mid; else lo = mid + 1;
            }
            iter.b = lo;
        }
        iter.seg = blockIdx.x;
    }

    if (warp == kConsumerWarps) {
        // =========================== producer warp ===========================
        const uint64_t policy = l2_evict_first_policy();
        uint32_t pos = 0;  // stream position (tiles issued by this CTA)
        Piece pc;
        while (iter.next(pc, a)) {
            const int h = pc.hh / nsub;
            const int32_t* trow = a.block_table + (int64_t)pc.b * a.max_blocks;
            // block id of tile t (one lane per tile, 32 at a time, next batch prefetched)
            auto fetch = [&](int t) -> int64_t {
                if (t >= pc.t1) return 0;
                const int32_t v = trow[(t * kTile) / a.block_size];
                if (v < 0 || v >= a.num_blocks) {
                    record_error(a.status, KVATTN_ERR_BAD_INDEX);
                    return 0;
                }
                return v;
            };
            int64_t blk_next = fetch(pc.t0 + lane);
            for (int base = pc.t0; base < pc.t1; base += 32) {
                const int64_t blk = blk_next;
                if (base + 32 < pc.t1) blk_next = fetch(base + 32 + lane);
                const int cnt = min(32, pc.t1 - base);
                // fp8 pages: kConsumerWarps tiles at a time, one per lane.  Their
                // stages are consecutive, freed by the consumer warps' concurrent
                // tiles, so the lanes' waits overlap and one instruction stream
                // issues all of their 4 KB copies (one lane issuing them in turn
                // could not keep HBM busy).  The 8 KB tiles of a bf16 cache go
                // one at a time: their shallower ring (two stages per consumer
                // warp) cannot afford a lane's copy waiting for its group's
                // slowest stage.
                constexpr int kIssue = kFP8 ? kConsumerWarps : 1;
                for (int j0 = 0; j0 < cnt; j0 += kIssue) {
                    const int j = j0 + lane;
                    const int64_t bj = __shfl_sync(0xffffffffu, blk, j & 31);
                    const bool aborted = *abort_flag != 0;
                    if (lane < kIssue && j < cnt && !aborted) {
                        const uint32_t my = pos + lane;
                        const uint32_t stage = my % stages, use = my / stages;
                        bool go = true;
                        if (use > 0) go = mbar_wait(&empty[stage], (use - 1) & 1, a.status);
                        if (!go) {
                            *abort_flag = 1;
                        } else {
                            const int tok = (base + j) * kTile;
                            const int nvalid = min(kTile, pc.len - tok);
                            const uint32_t bytes = (uint32_t)nvalid * kD * T::kE;
                            const int64_t row = (bj * a.hkv + h) * a.block_size + tok % a.block_size;
                            unsigned char* dst = ring + (size_t)stage * kStageB;
                            if constexpr (kFP8) {
                                // the fp8 page of these 16 tokens: K, V^T and scales, one copy
                                const int64_t page = row / kTile;
                                mbar_arrive_expect_tx(&full[stage], kF8Page);
                                bulk_load(dst, (const char*)a.k_pool + page * kF8Page, kF8Page, &full[stage], policy);
                            } else if constexpr (kMma) {
                                // whole 16-row pages (rows past the sequence end are
                                // masked out of S and zeroed in V by the consumer)
                                mbar_arrive_expect_tx(&full[stage], 2 * T::kTileBytes);
                                if constexpr (kRowBoxes) {
                                    for (int pnl = 0; pnl < 2; ++pnl) {
                                        tma_load_2d(dst + pnl * 2048, &maps.k, pnl * 64, (int)row, &full[stage], policy);
                                        tma_load_2d(dst + T::kTileBytes + pnl * 2048, &maps.v, pnl * 64, (int)row,
                                                    &full[stage], policy);
                                    }
                                } else {
                                    tma_load_4d(dst, &maps.k, 0, 0, 0, (int)(row >> 3), &full[stage], policy);
                                    tma_load_4d(dst + T::kTileBytes, &maps.v, 0, 0, 0, (int)(row >> 3), &full[stage],
                                                policy);
                                }
                            } else {
                                const char* ksrc = (const char*)a.k_pool + row * kD * T::kE;
                                const char* vsrc = (const char*)a.v_pool + row * kD * T::kE;
                                mbar_arrive_expect_tx(&full[stage], 2 * bytes);
                                bulk_load(dst, ksrc, bytes, &full[stage], policy);
                                bulk_load(dst + T::kTileBytes, vsrc, bytes, &full[stage], policy);
                            }
                        }
                    }
                    __syncwarp();
                    pos += min(kIssue, cnt - j0);
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
    const int M = T::mask(sub);          // XOR layout of this lane's partial scores
    const int hm = M / T::kTPG, tm = M % T::kTPG;
    constexpr int kMG = merge_heads<kGT, kFP8>();
    float2* pbuf = reinterpret_cast<float2*>(merge + (size_t)warp * kMG * (kD + 2)) + grp * T::kV;
    const int hq = a.hq;
    uint32_t pos = 0;
    Piece pc;

    while (iter.next(pc, a)) {
        const int h = pc.hh / nsub, hsub = pc.hh - h * nsub;
        const int ntiles = pc.t1 - pc.t0;
        const int qh0 = h * G + hsub * kGT;  // first query head of this segment
        float* mw = merge + (size_t)warp * kMG * (kD + 2);
        // Merge of the consumer warps' states for query heads h0 .. h0 + kMG - 1
        // of the segment (each warp has written its state for them into its
        // slot): the piece's result goes to out, or to its partial slot.
        auto merge_pass = [&](int h0) {
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
            const bool direct = pc.nslots == 1;
            if (h0 == 0 && tid == 0 && pc.slot == 0 && a.nslots) a.nslots[(int64_t)pc.b * HH + pc.hh] = pc.nslots;
            for (int e = tid; e < kMG * kD; e += kConsumerWarps * 32) {
                const int g = e / kD, d = e - g * kD;
                float Mx = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) Mx = fmaxf(Mx, merge[(w * kMG + g) * (kD + 2) + kD]);
                float num = 0.f, den = 0.f;
                if (Mx != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const float* mr = merge + (size_t)(w * kMG + g) * (kD + 2);
                        const float f = (mr[kD] == -INFINITY) ? 0.f : exp2f(mr[kD] - Mx);
                        num += f * mr[d];
                        den += f * mr[kD + 1];
                    }
                }
                const float o = den > 0.f ? num / den : 0.f;
                const int64_t qrow = (int64_t)pc.b * hq + qh0 + h0 + g;
                if (direct) {
                    if constexpr (kBF16)
                        reinterpret_cast<__nv_bfloat16*>(a.out)[qrow * kD + d] = __float2bfloat16_rn(o);
                    else
                        reinterpret_cast<float*>(a.out)[qrow * kD + d] = o;
                } else {
                    const int64_t prow = qrow * a.splits + pc.slot;
                    a.part_o[prow * kD + d] = o;
                    if (d == 0) {
                        a.part_ml[prow * 2] = Mx;
                        a.part_ml[prow * 2 + 1] = den;
                    }
                }
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
        };
        if constexpr (kFP8) {
            // ---- fp8 pages on the tensor cores (f16 operands; e4m3 codes are
            // exact in f16), tokens on the M axis and query heads on N, so
            // that no MMA row is padding: S^T = K Q^T is one m16n8k16 per
            // 16-dim step and O^T += V^T P^T one per 16 dims.  Row r of S^T
            // is token pi(r) = 4(r%8 / 2) + 2(r / 8) + r%2 of the page: lane
            // (g4, q4) then holds tokens rk0 = pi(g4) and rk1 = rk0 + 2, and
            // the dims of each k-step are permuted so that a lane's four K
            // values are one 32-bit word.  The C fragment of S^T, converted to
            // f16 P, becomes the B fragment of P^T by one 8x8 transpose per
            // half (movmatrix), which lands tokens 4q4 .. 4q4+3 of head g4 in
            // lane (g4, q4): one 32-bit word of the transposed V page holds a
            // lane's four tokens of one dim, the A operand of O^T += V^T P^T.
            // Q is scaled by 2^-4 into f16 range, the K scales multiply S per
            // token.  P carries each token's V scale over a lazy reference
            // vref (rescaled like the running max).
            const int g4 = lane >> 2, q4 = lane & 3;
            const int rk0 = (g4 >> 1) * 4 + (g4 & 1), rk1 = rk0 + 2;  // K rows (tokens) of this lane
            uint32_t qb[kD / 16][2];  // B fragment: head g4, dims 16kk + 4q4 .. 16kk + 4q4 + 3
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
                qb[kk][0] = qb[kk][1] = 0u;
                if (g4 < kGT) {
                    const uint2 w = *reinterpret_cast<const uint2*>(
                        reinterpret_cast<const __nv_bfloat16*>(a.q) + ((int64_t)pc.b * hq + qh0 + g4) * kD + kk * 16 +
                        4 * q4);
                    qb[kk][0] = pack_f16_rn(bf16lo(w.x) * 0.0625f, bf16hi(w.x) * 0.0625f);
                    qb[kk][1] = pack_f16_rn(bf16lo(w.y) * 0.0625f, bf16hi(w.y) * 0.0625f);
                }
            }
            // O^T fragments: dims 16m + g4 (o[m][0], o[m][1]) and 16m + 8 + g4
            // (o[m][2], o[m][3]) of heads 2q4 (even entries) and 2q4 + 1 (odd)
            float o[kD / 16][4];
#pragma unroll
            for (int m = 0; m < kD / 16; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
            float m_run[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};  // heads 2q4, 2q4 + 1
            float vref = 0.f, vinv = 0.f;
            const float sl2 = a.scale_log2 * 16.f;  // undoes the 2^-4 on Q
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
                const unsigned char* pg = ring + (size_t)stage * kStageB;
                const int tok0 = (pc.t0 + li) * kTile;
                const int nvalid = min(kTile, pc.len - tok0);
                float s[4] = {0.f, 0.f, 0.f, 0.f};  // S^T: (rk0, 2q4), (rk0, 2q4+1), (rk1, 2q4), (rk1, 2q4+1)
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t w0 =
                        *reinterpret_cast<const uint32_t*>(pg + rk0 * 128 + ((kk ^ f8_swz(rk0)) << 4) + 4 * q4);
                    const uint32_t w1 =
                        *reinterpret_cast<const uint32_t*>(pg + rk1 * 128 + ((kk ^ f8_swz(rk1)) << 4) + 4 * q4);
                    mma_f16_16816(s, e4m3x2_to_f16x2(w0), e4m3x2_to_f16x2(w1), e4m3x2_to_f16x2(w0 >> 16),
                                  e4m3x2_to_f16x2(w1 >> 16), qb[kk][0], qb[kk][1]);
                }
                // scores in log2 units
                const float* ksc = reinterpret_cast<const float*>(pg + kF8KsOff);
                const float* vsc = reinterpret_cast<const float*>(pg + kF8VsOff);
                const float k0 = ksc[rk0] * sl2, k1 = ksc[rk1] * sl2;
                float sv0 = vsc[rk0], sv1 = vsc[rk1];
                float x[4] = {s[0] * k0, s[1] * k0, s[2] * k1, s[3] * k1};
                uint32_t vmask = 0xffffffffu;  // bytes of this lane's V words that belong to valid tokens
                if (nvalid < kTile) {
                    if (rk0 >= nvalid) {
                        x[0] = x[1] = -INFINITY;
                        sv0 = 0.f;
                    }
                    if (rk1 >= nvalid) {
                        x[2] = x[3] = -INFINITY;
                        sv1 = 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (4 * q4 + j >= nvalid) vmask &= ~(0xffu << (8 * j));
                }
                // lazy references: the max of each head (raised when a tile
                // exceeds it by more than 2^8) and the V scale (when a tile's
                // is over 16x it); the tile's maxima over its 16 tokens are
                // only formed when some lane's own values call for a raise
                float l0 = fmaxf(x[0], x[2]), l1 = fmaxf(x[1], x[3]), lv = fmaxf(sv0, sv1);
                const bool raise = l0 > m_run[0] + 8.f || l1 > m_run[1] + 8.f || lv > vref * 16.f;
                if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
                    for (int sh = 4; sh < 32; sh <<= 1) {
                        l0 = fmaxf(l0, __shfl_xor_sync(0xffffffffu, l0, sh));
                        l1 = fmaxf(l1, __shfl_xor_sync(0xffffffffu, l1, sh));
                        lv = fmaxf(lv, __shfl_xor_sync(0xffffffffu, lv, sh));
                    }
                    float f0 = 1.f, f1 = 1.f;
                    if (l0 > m_run[0] + 8.f) {
                        f0 = m_run[0] == -INFINITY ? 0.f : fast_exp2(m_run[0] - l0);
                        lrun[0] *= f0;
                        m_run[0] = l0;
                    }
                    if (l1 > m_run[1] + 8.f) {
                        f1 = m_run[1] == -INFINITY ? 0.f : fast_exp2(m_run[1] - l1);
                        lrun[1] *= f1;
                        m_run[1] = l1;
                    }
                    if (lv > vref * 16.f) {
                        if (vref > 0.f) {
                            f0 *= vref / lv;
                            f1 *= vref / lv;
                        }
                        vref = lv;
                        vinv = 1.f / lv;
                    }
#pragma unroll
                    for (int m = 0; m < kD / 16; ++m) {
                        o[m][0] *= f0;
                        o[m][1] *= f1;
                        o[m][2] *= f0;
                        o[m][3] *= f1;
                    }
                }
                const float p0 = fast_exp2(x[0] - m_run[0]), p1 = fast_exp2(x[1] - m_run[1]);
                const float p2 = fast_exp2(x[2] - m_run[0]), p3 = fast_exp2(x[3] - m_run[1]);
                lrun[0] += p0 + p2;
                lrun[1] += p1 + p3;
                const float c0 = sv0 * vinv, c1 = sv1 * vinv;
                // P^T B fragment: head g4, tokens 4q4, 4q4+1 (pb0) and 4q4+2, 4q4+3 (pb1)
                const uint32_t pb0 = movmatrix_trans(pack_f16_rn(p0 * c0, p1 * c0));
                const uint32_t pb1 = movmatrix_trans(pack_f16_rn(p2 * c1, p3 * c1));
                // V^T words: dims 16m + g4 and 16m + 8 + g4, tokens 4q4 .. 4q4+3
                // (stale tokens zeroed: 0 * NaN)
                const unsigned char* vt = pg + kF8VOff + g4 * 16 + 4 * q4;
#pragma unroll
                for (int m = 0; m < kD / 16; ++m) {
                    const uint32_t wa = *reinterpret_cast<const uint32_t*>(vt + m * 256) & vmask;
                    const uint32_t wb = *reinterpret_cast<const uint32_t*>(vt + m * 256 + 128) & vmask;
                    mma_f16_16816(o[m], e4m3x2_to_f16x2(wa), e4m3x2_to_f16x2(wb), e4m3x2_to_f16x2(wa >> 16),
                                  e4m3x2_to_f16x2(wb >> 16), pb0, pb1);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
            }
            pos += ntiles;
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) {
                lrun[0] += __shfl_xor_sync(0xffffffffu, lrun[0], sh);
                lrun[1] += __shfl_xor_sync(0xffffffffu, lrun[1], sh);
            }
            __syncwarp();
#pragma unroll
            for (int h0 = 0; h0 < kGT; h0 += kMG) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int hd = 2 * q4 + e;
                    if (hd >= h0 && hd < h0 + kMG && hd < kGT) {
                        float* mr = mw + (hd - h0) * (kD + 2);
#pragma unroll
                        for (int m = 0; m < kD / 16; ++m) {
                            mr[16 * m + g4] = o[m][e] * vref;
                            mr[16 * m + 8 + g4] = o[m][2 + e] * vref;
                        }
                        if (g4 == 0) {
                            mr[kD] = m_run[e];
                            mr[kD + 1] = lrun[e];
                        }
                    }
                }
                merge_pass(h0);
            }
        } else if constexpr (kMma) {
            // ---- tensor-core path: S = Q K^T and O += P V as m16n8k16 MMAs
            // with the query heads as rows (rows kGT..15 zero), so that the
            // accumulator fragments of S are the A fragments of P.V
            const int g4 = lane >> 2, q4 = lane & 3;  // fragment row, column pair
            const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix and row this lane addresses
            constexpr int gs = kRowBoxes ? 1024 : 2048, ps = kRowBoxes ? 2048 : 1024;  // group, panel strides
            uint32_t qa[kD / 16][2];                  // Q rows g4: columns 2q4.. and 8+2q4.. of each k-step
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
                qa[kk][0] = qa[kk][1] = 0u;
                if (g4 < kGT) {
                    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                        reinterpret_cast<const __nv_bfloat16*>(a.q) + ((int64_t)pc.b * hq + qh0 + g4) * kD + kk * 16);
                    qa[kk][0] = qrow[q4];
                    qa[kk][1] = qrow[4 + q4];
                }
            }
            float o[kD / 8][2];  // rows 0..7 of each 16 x 8 output fragment (rows 8..15 are padding)
#pragma unroll
            for (int nd = 0; nd < kD / 8; ++nd) o[nd][0] = o[nd][1] = 0.f;
            float m_run = -INFINITY, lrun = 0.f;
            const float sl2 = a.scale_log2;
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
                unsigned char* kst = ring + (size_t)stage * T::kStageBytes;
                unsigned char* vst = kst + T::kTileBytes;
                const int tok0 = (pc.t0 + li) * kTile;
                const int nvalid = min(kTile, pc.len - tok0);
                // page rows past the sequence end are stale: masked out of S,
                // zeroed in V (their p is 0, but 0 * NaN would be NaN)
                if (nvalid < kTile) {
                    for (int idx = lane; idx < (kTile - nvalid) * 16; idx += 32) {
                        const int row = nvalid + (idx >> 4), c = idx & 15;
                        *reinterpret_cast<uint4*>(vst + (row >> 3) * gs + (c >> 3) * ps + (row & 7) * 128 +
                                                  (c & 7) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    __syncwarp();
                }
                // 16-byte chunk c of row r at chunk (c ^ r) of its 128 B (r = row mod 8)
                const uint32_t kb = smem_addr(kst), vb = smem_addr(vst);
                float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};  // tokens 0-7, 8-15 (rows 0..7 of the fragments)
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    // matrices (tokens 0-7, chunk 2kk), (0-7, 2kk+1), (8-15, 2kk), (8-15, 2kk+1)
                    const int c = 2 * kk + (mi & 1), grp = mi >> 1;
                    uint32_t b[4];
                    ldmatrix_x4(b, kb + grp * gs + (c >> 3) * ps + rr * 128 + (((c & 7) ^ rr) << 4));
                    mma_bf16_16816_top(s0, qa[kk][0], qa[kk][1], b[0], b[1]);
                    mma_bf16_16816_top(s1, qa[kk][0], qa[kk][1], b[2], b[3]);
                }
                // row g4: tokens 2q4, 2q4+1 (s0) and 8+2q4, 9+2q4 (s1), in log2 units
                float x[4] = {s0[0] * sl2, s0[1] * sl2, s1[0] * sl2, s1[1] * sl2};
                if (2 * q4 >= nvalid) x[0] = -INFINITY;
                if (2 * q4 + 1 >= nvalid) x[1] = -INFINITY;
                if (2 * q4 + 8 >= nvalid) x[2] = -INFINITY;
                if (2 * q4 + 9 >= nvalid) x[3] = -INFINITY;
                float tmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
                // reference max, raised only when a tile's max exceeds it by
                // more than 2^8 (p <= 256, rare rescale of O)
                if (tmax > m_run + 8.f) {
                    const float alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - tmax);
                    m_run = tmax;
                    lrun *= alpha;
#pragma unroll
                    for (int nd = 0; nd < kD / 8; ++nd) {
                        o[nd][0] *= alpha;
                        o[nd][1] *= alpha;
                    }
                }
                const float p0 = fast_exp2(x[0] - m_run), p1 = fast_exp2(x[1] - m_run);
                const float p2 = fast_exp2(x[2] - m_run), p3 = fast_exp2(x[3] - m_run);
                lrun += (p0 + p1) + (p2 + p3);
                const uint32_t pa0 = pack_bf16_rn(p0, p1), pa2 = pack_bf16_rn(p2, p3);
#pragma unroll
                for (int nd2 = 0; nd2 < kD / 16; ++nd2) {
                    // V^T fragments: matrices (tokens 0-7, chunk 2nd2), (8-15, 2nd2), (0-7, 2nd2+1), (8-15, 2nd2+1)
                    const int c = 2 * nd2 + (mi >> 1), grp = mi & 1;
                    uint32_t b[4];
                    ldmatrix_x4_trans(b, vb + grp * gs + (c >> 3) * ps + rr * 128 + (((c & 7) ^ rr) << 4));
                    mma_bf16_16816_top(o[2 * nd2], pa0, pa2, b[0], b[1]);
                    mma_bf16_16816_top(o[2 * nd2 + 1], pa0, pa2, b[2], b[3]);
                }
                if (nvalid < kTile) fence_async_smem();  // zeroed rows before the next copy into this stage
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
            }
            pos += ntiles;
            lrun += __shfl_xor_sync(0xffffffffu, lrun, 1);
            lrun += __shfl_xor_sync(0xffffffffu, lrun, 2);
            __syncwarp();
#pragma unroll
            for (int h0 = 0; h0 < kGT; h0 += kMG) {
                if (g4 >= h0 && g4 < h0 + kMG) {
                    float* mr = mw + (g4 - h0) * (kD + 2);
#pragma unroll
                    for (int nd = 0; nd < kD / 8; ++nd)
                        *reinterpret_cast<float2*>(mr + nd * 8 + 2 * q4) = make_float2(o[nd][0], o[nd][1]);
                    if (q4 == 0) {
                        mr[kD] = m_run;
                        mr[kD + 1] = lrun;
                    }
                }
                merge_pass(h0);
            }
        } else {

        // query slice of this lane (head g^hm in slot g), pre-scaled by scale*log2(e)
        uint64_t q2[kGT][T::kP];
#pragma unroll
        for (int g = 0; g < kGT; ++g) {
            const char* qrow = (const char*)a.q + ((int64_t)pc.b * hq + qh0 + (g ^ hm)) * kD * T::kE;
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
        const int my_g = M / T::kTPG;  // the one head whose scores this lane ends up with

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
            const int tok0 = (pc.t0 + li) * kTile;
            const int nvalid = min(kTile, pc.len - tok0);

            // ---- partial scores, slot (g, t) holding head g^hm, token t^tm
            float sc[T::kV];
#pragma unroll
            for (int t = 0; t < T::kTPG; ++t) {
                const int row = grp * T::kTPG + (t ^ tm);
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
            Bfly<T::kV, T::kLPG / 2>::run(sc);

            // ---- this lane's scores (logical index M + r): mask, group max
            float bmax = -INFINITY;
#pragma unroll
            for (int r = 0; r < T::kR; ++r) {
                const int tt = (M + r) % T::kTPG;
                if (grp * T::kTPG + tt >= nvalid) sc[r] = -INFINITY;
                bmax = fmaxf(bmax, sc[r]);
            }
#pragma unroll
            for (int o = T::kBW / 2; o >= 1; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
            float mnew[kGT], alpha[kGT];
            bool grow = false;
#pragma unroll
            for (int g = 0; g < kGT; ++g) {
                const float tmx = __shfl_sync(0xffffffffu, bmax, grp * T::kLPG + g * T::kBW);
                mnew[g] = fmaxf(m[g], tmx);
                alpha[g] = (mnew[g] == -INFINITY) ? 1.f : exp2f(m[g] - mnew[g]);
                grow |= mnew[g] != m[g];
            }
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
            // ---- share probabilities inside the group, as (p, p) pairs
#pragma unroll
            for (int r = 0; r < T::kR; ++r) pbuf[M + r] = make_float2(sc[r], sc[r]);
            __syncwarp();
            // ---- weighted V
            const uint64_t* pb2 = reinterpret_cast<const uint64_t*>(pbuf);
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
                        const uint64_t p2 = pb2[g * T::kTPG + t];   // (p, p)
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
            float Mx = m[g];
#pragma unroll
            for (int o = T::kLPG; o < 32; o <<= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));
            const float f = (m[g] == -INFINITY) ? 0.f : exp2f(m[g] - Mx);
            l *= f;
            const uint64_t f2 = pk(f, f);
#pragma unroll
            for (int i = 0; i < T::kP; ++i) acc[g][i] = fmul2(acc[g][i], f2);
#pragma unroll
            for (int o = T::kLPG; o < 32; o <<= 1) {
                l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
                for (int i = 0; i < T::kP; ++i) acc[g][i] = fadd2(acc[g][i], __shfl_xor_sync(0xffffffffu, acc[g][i], o));
            }
            m[g] = Mx;
            lsum[g] = l;
        }
        // ---- write this warp's state (over its own probability buffer), merge the warps
        __syncwarp();
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
        merge_pass(0);
        }  // CUDA-core path
    }
}

// Merge the partial slots of the segments that were cut into several pieces.
template <bool kBF16, int kD>
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__ DecodeArgs a, const int gt)
{
    pdl_wait();
    const int wid = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (wid >= a.batch * a.hq) return;
    const int b = wid / a.hq, qh = wid - b * a.hq;
    const int G = a.hq / a.hkv, nsub = G / gt;
    const int hh = (qh / G) * nsub + (qh % G) / gt;
    const int ns = a.nslots[(int64_t)b * a.hkv * nsub + hh];
    if (ns <= 1) return;
    constexpr int kDL = kD / 32;
    const float* ml = a.part_ml + (int64_t)wid * a.splits * 2;
    float M = -INFINITY;
    for (int c = 0; c < ns; ++c) M = fmaxf(M, ml[2 * c]);
    float acc[kDL];
#pragma unroll
    for (int i = 0; i < kDL; ++i) acc[i] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
        for (int c = 0; c < ns; ++c) {
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

template <bool kBF16, int kD, int kGT, bool kMma, bool kRowBoxes = false, bool kFP8 = false>
kvattn_status run(const DecodeArgs& a, cudaStream_t s)
{
    constexpr int kStageB = stage_bytes<kBF16, kD, kGT, kFP8>();
    PageMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if constexpr (kMma && !kFP8) {
        const int64_t rows = a.num_blocks * a.hkv * a.block_size;
        if (!pool_maps(a.k_pool, a.v_pool, rows, kRowBoxes, &maps.k, &maps.v)) return KVATTN_ERR_CUDA;
    }
    // Ring depth: as many stages (up to 64 KB of them) as leave room for
    // ctas_per_sm CTAs per SM, counting the per-block reserved shared memory.
    DeviceSmem dsm;
    if (!device_smem(&dsm)) return KVATTN_ERR_CUDA;
    const int smem_sm = dsm.per_sm, smem_reserved = dsm.reserved;
    // The depth must be a multiple of the consumer-warp count: then stage s is
    // always consumed by warp s % kConsumerWarps, in order, which keeps every
    // mbarrier wait at most one phase away from the phase it names (parity
    // waits cannot tell phase u from phase u - 2).
    const int fixed = shared_layout<kBF16, kD, kGT, kFP8>(0, a.batch).bytes + 1024;  // + base alignment slack
    const int per_stage = kStageB + 16;  // + two mbarriers
    const int budget = smem_sm / ctas_per_sm<kMma, kFP8>() - smem_reserved - fixed;
    int stages = std::min(65536 / kStageB, budget / per_stage);
    stages = std::max(kConsumerWarps, stages / kConsumerWarps * kConsumerWarps);
    const SharedLayout SL = shared_layout<kBF16, kD, kGT, kFP8>(stages, a.batch);
    const int smem_bytes = SL.bytes + 1024;
    auto kern = decode_split_kernel<kBF16, kD, kGT, kMma, kRowBoxes, kFP8>;
    static SmemLimit limit;
    if (limit.ensure(reinterpret_cast<const void*>(kern), smem_bytes) != cudaSuccess) return KVATTN_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem_bytes) != cudaSuccess)
        return KVATTN_ERR_CUDA;
    per_sm = std::max(1, per_sm);
    const int grid = num_sms() * per_sm;
    cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kThreads), smem_bytes, s, a, maps, stages);
    if (e != cudaSuccess) return KVATTN_ERR_CUDA;
    if (a.splits > 1) {
        const int warps = a.batch * a.hq;
        e = launch_pdl(decode_combine_kernel<kBF16, kD>, dim3((warps + 3) / 4), dim3(128), 0, s, a, kGT);
    }
    return cuda_status(e);
}

}  // namespace

DecodePlan decode_plan(int32_t batch, int32_t hkv, int32_t group, int32_t max_seq_len, int32_t splits)
{
    DecodePlan p;
    const int max_tiles = std::max(1, (max_seq_len + kTile - 1) / kTile);
    if (splits > 0) {
        p.slots = splits;
    } else {
        // Flat decomposition with at most `slots` pieces per segment: a CTA
        // range holds ceil(total / grid) tiles, and the piece cap forces at
        // least ceil(max_tiles / (slots - 1)) per range.  With lengths spread
        // up to max_seq_len the total is about batch*segments*max_tiles/2, so
        // slots - 1 >= 4 * grid / (batch * segments) keeps the cap inactive
        // with a factor-2 margin.
        const int nsub = group > 4 ? group / 4 : 1;
        const int64_t segs = std::max<int64_t>(1, (int64_t)batch * hkv * nsub);
        const int64_t grid = (int64_t)num_sms() * 3;
        const int64_t want = 1 + (4 * grid + segs - 1) / segs;
        p.slots = (int32_t)std::max<int64_t>(3, std::min<int64_t>(16, want));
    }
    p.slots = std::min(p.slots, max_tiles + 1);
    if (p.slots < 1) p.slots = 1;
    return p;
}

kvattn_status launch_decode(const DecodeArgs& a, cudaStream_t s)
{
    const int G = a.hq / a.hkv;
    const bool bf16 = a.dtype == KVATTN_BF16;
    const int gt = G >= 4 ? 4 : G;
    if (a.fp8) {  // fp8 pages: the tensor-core path, every head of the group in one segment
        if (!(bf16 && a.d == 128 && (G == 4 || G == 8) && a.block_size % 16 == 0)) return KVATTN_ERR_UNSUPPORTED;
        return G == 8 ? run<true, 128, 8, true, false, true>(a, s) : run<true, 128, 4, true, false, true>(a, s);
    }
    // bf16, D = 128, groups of 4 or 8 query heads per KV head: QK and PV on the
    // tensor cores with the group's heads as rows 0..G-1 of the MMA fragments,
    // so every page is read once per KV head (tensor-map row coordinates are
    // 32-bit)
    if (bf16 && a.d == 128 && (G == 4 || G == 8) && a.num_blocks * a.hkv * a.block_size < ((int64_t)1 << 31)) {
        if (G == 8)
            return a.block_size % 16 == 0 ? run<true, 128, 8, true, false>(a, s) : run<true, 128, 8, true, true>(a, s);
        return a.block_size % 16 == 0 ? run<true, 128, 4, true, false>(a, s) : run<true, 128, 4, true, true>(a, s);
    }
#define KVATTN_DECODE_CASE(BF, DD, GG) \
    if (bf16 == BF && a.d == DD && gt == GG) return run<BF, DD, GG, false>(a, s);
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
