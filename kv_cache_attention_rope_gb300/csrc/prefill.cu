// Chunked-prefill causal attention on the tcgen05 tensor cores.
//
// What it computes ("From-scratch AI inference engine" page, sections 3.1,
// 3.3 and 3.4): for chunk c with prefix P (tokens already cached before the
// chunk) and query row r of the chunk at absolute position P + r,
//     out[r] = softmax_{k <= P + r}(q[r] . K[k] * scale) V[k]
// over the keys of the chunk's sequence in the paged cache, which already
// holds the chunk's own keys.  The online softmax (running max and sum, the
// accumulated output rescaled when the max grows) tiles the key axis.
//
// How (GB300 design): persistent CTAs, one per SM, each running a sorted
// share of the work items (chunk, 256 query rows, query head); an item's rows
// are two 128-row tiles A and B that share one K/V stream:
//  - warp 0 (one lane) streams with TMA tensor copies: both 128 x 128 bf16 Q
//    tiles once, then 128-key K and V tiles (two stages each), each gathered
//    as eight 16-token pages of the KV head straight from the block table,
//    one 4 KB copy per page, issued by the page's own lane (a single lane
//    issuing the eight copies one after another was the slowest step of the
//    whole pipeline), 128-byte swizzled (the layout the MMA reads).
//    A K/V stage is laid out [8-key group][64-column panel][8 keys][128 B]:
//    a page is then one contiguous 4 KB box of a 4-D view of the pool, and
//    both MMA operand descriptors still see uniform strides (2 KB between
//    8-key groups, 1 KB between panels).  Halving the number of copies (one
//    4 KB box instead of two 2 KB boxes per page) cut the kernel's time by a
//    quarter: with 32 small copies per tile the stream was bound by copies
//    issued, not by bytes.
//  - warp 1 (one elected lane) issues the MMAs: S_x = Q_x K^T (M = N = 128, K = 128,
//    both operands in shared memory) and O_x += P_x V (P_x read from TMEM,
//    V an MN-major shared-memory operand), x = A, B.  TMEM (512 columns)
//    holds S_A, S_B, O_A, O_B; P_x (bf16, 64 columns) overwrites the first
//    half of S_x once the softmax has read it.  Taking P from TMEM halves the
//    shared-memory operand traffic of P.V, which at N = 128 would otherwise
//    saturate shared-memory bandwidth before the tensor core.
//    Issue order per KV tile j: PV_A(j) S_A(j+1) PV_B(j) S_B(j+1): tensor
//    operations of one thread run in issue order, so S_A(j+1) overwrites
//    S_A's columns only after PV_A(j) has read P_A(j) from them, and while
//    the softmax of tile A works on S_A(j+1) the tensor core runs PV_B(j) and
//    S_B(j+1) (ping-pong).  Completion is signalled with tcgen05.commit on
//    mbarriers; a commit covers every earlier MMA of the thread, so when
//    S_x(j+1) is reported done, PV_x(j) is too and O_x may be rescaled.
//  - warps 2-9 run the softmax of whichever tile is due, two threads per
//    query row (= TMEM lane), one per 64-column half: load the half row of S
//    from TMEM, apply the causal mask on diagonal tiles, agree on the row max
//    with the other half through shared memory, keep the running max (raised
//    only when it grows by more than 2^8, which bounds p by 256 and keeps the
//    O rescale rare), write P as bf16 into TMEM for the next MMA, and finally
//    read O, divide by the row sum and store bf16.
//  - Every wait is bounded (1 s): a timeout records KVATTN_ERR_TIMEOUT, the
//    roles stop waiting, drain their in-flight copies and MMAs, free TMEM and
//    return.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "kvattn_tc.cuh"

namespace kvattn {
namespace {

constexpr int kBM = 128;      // query rows per tile (two tiles per CTA: A and B)
constexpr int kBN = 128;      // keys per KV tile
constexpr int kPage = 16;     // tokens per TMA copy of one block
constexpr int kThreads = 320; // warp 0 TMA, warp 1 MMA, warps 2-5 softmax A, warps 6-9 softmax B
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kPanel = kBM * 128;          // 16 KB: 128 rows x 64 columns (one 128-byte swizzle panel of Q)
constexpr int kNumBars = 2 + 2 * kKStages + 2 * kVStages + 2 + 2 + 2 + 1;
constexpr int kMaxPairs = 1024;            // more (chunk, 256-row) pairs than this: unsorted order
static_assert(kNumBars * 8 + 8 <= 256, "barriers, TMEM address and abort flag fit before the exchange area");

// Shared-memory geometry for head dim kD (64 or 128): a row of Q, K or V is
// kD / 64 panels of 128 bytes; a K/V stage is [8-key group][panel][8 keys]
// [128 B], so a 16-token page is one contiguous block of the stage.
template <int kD>
struct Geo {
    static constexpr int kPanels = kD / 64;
    static constexpr int kTileBytes = kBM * kD * 2;  // a Q tile, a K stage or a V stage (32 KB at D = 128)
    static constexpr int kGroup = 8 * kD * 2;        // one 8-key group of a stage (all panels)
    static constexpr int kPageBytes = kPage * kD * 2; // one 16-token page of K or V (4 KB at D = 128)
    static constexpr int kOffQ = 0;                   // Q_A, Q_B
    static constexpr int kOffK = 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
    static constexpr int kOffX = kOffBar + 256;  // softmax exchange: row maxima [2][2][128], row sums [2][2][128] (fp32)
    static constexpr int kOffOrder = kOffX + 4096;  // work order: sorted pairs, tiles per pair (int32)
    static constexpr int kOffStage = (kOffOrder + 2 * kMaxPairs * 4 + 1023) / 1024 * 1024;  // output staging, 2 KB per softmax warp
    static constexpr int kSmemBytes = kOffStage + 8 * 2048 + 1024;  // + slack to align the base to 1 KB
    static_assert(kD == 64 || kD == 128, "head dim");
};

struct Maps {
    CUtensorMap q;  // 3-D: (D, Hq, total_q), box (64, 1, 128)
    CUtensorMap o;  // 3-D: (D, Hq, total_q), box (32, 1, 32), 64-byte swizzle (output stores)
    CUtensorMap k;  // 4-D: (64 columns, 8 rows, 2 panels, rows / 8), box (64, 8, 2, 2)
    CUtensorMap v;
};

struct Bars {
    uint64_t* q_full;
    uint64_t* q_empty;  // every S MMA of the current item is done
    uint64_t* k_full;   // [kKStages]
    uint64_t* k_empty;  // [kKStages]
    uint64_t* v_full;   // [kVStages]
    uint64_t* v_empty;  // [kVStages]
    uint64_t* s_full;   // [2]: tile A, tile B
    uint64_t* p_full;   // [2]
    uint64_t* o_done;   // [2]: the last P.V of the tile has completed
    uint64_t* drain;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status)
{
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, status)) return true;
    *abort_flag = 1;
    return false;
}

// 2^x with the hardware approximation (ex2.approx.ftz: a few ulp relative
// error, far below the bf16 rounding P goes through); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Whole-warp wait: every lane waits, the warp agrees (tcgen05.ld/st that
// follow are warp-collective, so a partial warp must never reach them).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status)
{
    const bool ok = wait_or_abort(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// Named barrier `id` over `nthreads` threads that also returns the AND of
// every participant's `v` (bar.red.and).
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool v)
{
    uint32_t res;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(res)
        : "r"((uint32_t)v), "r"(id), "r"(nthreads)
        : "memory");
    return res != 0;
}

// One lane of the (converged) warp is elected: it alone issues tensor-core
// instructions, while the warp's uniform values stay in uniform registers.
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred = 0;
    asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(pred));
    return pred != 0;
}

// One work item: query rows [256 qt, 256 qt + 256) of chunk c, query head j,
// as tiles A (first 128 rows) and B (next 128) against the same K/V stream.
struct Item {
    int c, j, h;      // chunk, query head, KV head
    int seq_len;      // prefix + chunk length
    int rows;         // valid rows of the 256
    int row0;         // first q row (token index)
    int pos0;         // absolute position of row 0
    int n_kv;         // 128-key tiles (0: nothing to do)
};

// Tiles of the (chunk, 256-row block) pair: the key range row 255 (or the
// last row) sees; 0 when the block is past the chunk's end or the chunk's
// metadata is out of range (recorded by make_item).
__device__ __forceinline__ int pair_tiles(const PrefillArgs& a, int n_qt, int pair)
{
    const int c = pair / n_qt, qt = pair % n_qt;
    const int q0 = a.cu_q_lens[c], qlen = a.cu_q_lens[c + 1] - q0, P = a.prefix_lens[c];
    if (qt * 2 * kBM >= qlen) return 0;
    if (qlen < 0 || P < 0 || qlen > a.max_q_len || q0 < 0 || q0 + qlen > a.total_q ||
        (int64_t)(P + qlen) > (int64_t)a.max_blocks * a.block_size)
        return 0;
    const int rows = min(2 * kBM, qlen - qt * 2 * kBM);
    return (P + qt * 2 * kBM + rows - 1) / kBN + 1;
}

__device__ __forceinline__ Item make_item(const PrefillArgs& a, int n_qt, int pair, int j, bool report)
{
    Item it;
    it.c = pair / n_qt;
    const int qt = pair % n_qt;
    it.j = j;
    it.h = j / (a.hq / a.hkv);
    const int q0 = a.cu_q_lens[it.c], qlen = a.cu_q_lens[it.c + 1] - q0, P = a.prefix_lens[it.c];
    it.seq_len = P + qlen;
    it.n_kv = 0;
    it.rows = it.row0 = it.pos0 = 0;
    if (qt * 2 * kBM >= qlen) return it;  // nothing to do
    if (qlen < 0 || P < 0 || qlen > a.max_q_len || q0 < 0 || q0 + qlen > a.total_q ||
        (int64_t)it.seq_len > (int64_t)a.max_blocks * a.block_size) {
        if (report) record_error(a.status, KVATTN_ERR_BAD_INDEX);
        return it;
    }
    it.rows = min(2 * kBM, qlen - qt * 2 * kBM);
    it.row0 = q0 + qt * 2 * kBM;
    it.pos0 = P + qt * 2 * kBM;
    it.n_kv = (it.pos0 + it.rows - 1) / kBN + 1;
    return it;
}

// Persistent CTAs (one per SM).  Work items are (pair, head) with pairs in
// descending order of KV tiles (every CTA ranks them identically in shared
// memory; ties by index), heads innermost, so the query heads of one KV head
// run side by side and share its pages through L2.  CTA k takes, in round r,
// item r G + k for even r and r G + G - 1 - k for odd r (G CTAs): a snake
// over the sorted list, which balances the long items against the short
// ones without a global counter.  Pipeline state (stages, phases) runs on
// across items, so the next item's Q, K, V and first S overlap the current
// item's last tiles and epilogue.
template <int kHD>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ Maps maps, const int n_qt)
{
    pdl_wait();
    using GE = Geo<kHD>;
    constexpr int kTileBytes = GE::kTileBytes, kPageBytes = GE::kPageBytes, kGroup = GE::kGroup;
    constexpr int kOffQ = GE::kOffQ, kOffK = GE::kOffK, kOffV = GE::kOffV;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + GE::kOffBar);
    Bars B;
    {
        uint64_t* b = bar;
        B.q_full = b; b += 1;
        B.q_empty = b; b += 1;
        B.k_full = b; b += kKStages;
        B.k_empty = b; b += kKStages;
        B.v_full = b; b += kVStages;
        B.v_empty = b; b += kVStages;
        B.s_full = b; b += 2;
        B.p_full = b; b += 2;
        B.o_done = b; b += 2;
        B.drain = b;
    }
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* order = reinterpret_cast<int*>(smem + GE::kOffOrder);  // sorted pairs
    int* plen = order + kMaxPairs;                          // tiles per pair

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_pairs = a.num_chunks * n_qt;
    const bool sorted = n_pairs <= kMaxPairs;
    if (sorted) {
        for (int i = threadIdx.x; i < n_pairs; i += kThreads) plen[i] = pair_tiles(a, n_qt, i);
    }
    if (threadIdx.x == 0) {
        mbar_init(B.q_full, 1);
        mbar_init(B.q_empty, 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&B.k_full[s], 1);
            mbar_init(&B.k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&B.v_full[s], 1);
            mbar_init(&B.v_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&B.s_full[x], 1);
            mbar_init(&B.p_full[x], 256);
            mbar_init(&B.o_done[x], 1);
        }
        mbar_init(B.drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    __syncthreads();
    if (sorted) {  // rank = pairs with more tiles, or as many and a smaller index
        for (int i = threadIdx.x; i < n_pairs; i += kThreads) {
            const int li = plen[i];
            int rank = 0;
            for (int q = 0; q < n_pairs; ++q) {
                const int lq = plen[q];
                rank += (lq > li) || (lq == li && q < i);
            }
            order[rank] = i;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;  // S_A at +0, S_B at +128, O_A at +256, O_B at +384
    const int n_items = n_pairs * a.hq;
    const int G = gridDim.x, k_cta = blockIdx.x;
    // i-th item of this CTA's sequence (-1 past the end)
    auto item_index = [&](int r) -> int {
        const int i = r * G + ((r & 1) ? G - 1 - k_cta : k_cta);
        return i < n_items ? i : -1;
    };
    auto item_at = [&](int i, bool report) -> Item {
        const int pr = i / a.hq;
        return make_item(a, n_qt, sorted ? order[pr] : pr, i % a.hq, report);
    };

    if (warp == 0) {
        // ================================ TMA producer ================================
        const uint64_t pol_q = l2_evict_first_policy();
        const uint64_t pol_kv = l2_evict_normal_policy();
        if (lane == 0) {
            tma_prefetch_map(&maps.q);
            tma_prefetch_map(&maps.k);
            tma_prefetch_map(&maps.v);
        }
        int g = 0, ii = 0;    // tiles and items started so far (this CTA)
        int kg = 0, vg = 0;   // tiles whose K / V copies are armed
        bool go = true;
        for (int r = 0; go; ++r) {
            const int i = item_index(r);
            if (i < 0) break;
            const Item it = item_at(i, lane == 0);
            if (it.n_kv == 0) continue;
            // Q tiles: free once every S MMA of the previous item is done
            if (lane == 0) {
                go = ii > 0 ? wait_or_abort(B.q_empty, (ii - 1) & 1, abort_flag, a.status) : !*abort_flag;
                if (go) {
                    mbar_arrive_expect_tx(B.q_full, 2 * kTileBytes);
                    for (int x = 0; x < 2; ++x)
                        for (int p = 0; p < GE::kPanels; ++p)
                            tma_load_3d(smem + kOffQ + x * kTileBytes + p * kPanel, &maps.q, 64 * p, it.j,
                                        it.row0 + x * kBM, B.q_full, pol_q);
                }
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            if (!go) break;
            ++ii;
            const int32_t* trow = a.block_table + (int64_t)it.c * a.max_blocks;
            // lane p < 8 loads the block id of page p of tile t (keys 128t + 16p ..)
            auto fetch = [&](int t) -> int32_t {
                const int key0 = t * kBN + lane * kPage;
                return (lane < kBN / kPage && t < it.n_kv && key0 < it.seq_len) ? trow[key0 / a.block_size] : -1;
            };
            int32_t blk_next = fetch(0);
            for (int t = 0; t < it.n_kv; ++t, ++g) {
                const int32_t blk = blk_next;
                blk_next = fetch(t + 1);  // in flight while this tile is issued
                int y = 0;
                bool have = false;
                const int key0 = t * kBN + lane * kPage;
                if (lane < kBN / kPage && key0 < it.seq_len) {
                    if (blk < 0 || blk >= a.num_blocks) {
                        record_error(a.status, KVATTN_ERR_BAD_INDEX);
                    } else {
                        y = (int)(((int64_t)blk * a.hkv + it.h) * a.block_size + key0 % a.block_size);
                        have = true;
                    }
                }
                const unsigned pages = __ballot_sync(0xffffffffu, have);
                const uint32_t bytes = (uint32_t)__popc(pages) * (uint32_t)kPageBytes;
                // K stage g % kKStages: free once S_A and S_B of tile g - kKStages are done
                const int ks = g % kKStages;
                if (lane == 0) {
                    go = g >= kKStages ? wait_or_abort(&B.k_empty[ks], ((g / kKStages) - 1) & 1, abort_flag, a.status)
                                       : !*abort_flag;
                    if (go) mbar_arrive_expect_tx(&B.k_full[ks], bytes);
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) break;
                if (have) {
                    if constexpr (kHD == 128)
                        tma_load_4d(smem + kOffK + ks * kTileBytes + lane * kPageBytes, &maps.k, 0, 0, 0, y >> 3,
                                    &B.k_full[ks], pol_kv);
                    else
                        tma_load_2d(smem + kOffK + ks * kTileBytes + lane * kPageBytes, &maps.k, 0, y, &B.k_full[ks],
                                    pol_kv);
                }
                kg = g + 1;
                // V stage g % kVStages: free once PV_A and PV_B of tile g - kVStages are done
                const int vs = g % kVStages;
                if (lane == 0) {
                    go = g >= kVStages ? wait_or_abort(&B.v_empty[vs], ((g / kVStages) - 1) & 1, abort_flag, a.status)
                                       : !*abort_flag;
                    if (go) mbar_arrive_expect_tx(&B.v_full[vs], bytes);
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) break;
                if (have) {
                    if constexpr (kHD == 128)
                        tma_load_4d(smem + kOffV + vs * kTileBytes + lane * kPageBytes, &maps.v, 0, 0, 0, y >> 3,
                                    &B.v_full[vs], pol_kv);
                    else
                        tma_load_2d(smem + kOffV + vs * kTileBytes + lane * kPageBytes, &maps.v, 0, y, &B.v_full[vs],
                                    pol_kv);
                }
                vg = g + 1;
            }
        }
        // After an abort, let every armed copy land before the CTA can exit.
        if (lane == 0 && *abort_flag) {
            for (int t = max(0, kg - kKStages); t < kg; ++t)
                mbar_wait(&B.k_full[t % kKStages], (t / kKStages) & 1, a.status);
            for (int t = max(0, vg - kVStages); t < vg; ++t)
                mbar_wait(&B.v_full[t % kVStages], (t / kVStages) & 1, a.status);
            if (ii > 0) mbar_wait(B.q_full, (ii - 1) & 1, a.status);
        }
    } else if (warp == 1) {
        // ================================ MMA issuer =================================
        // The whole warp runs the schedule (waits agreed by the warp) and one
        // elected lane issues.  Operand descriptors are built once: a stage or
        // k-step only adds (byte offset >> 4) to the start-address field, which
        // cannot carry out of it (shared-memory offsets stay below 256 KB).  A
        // lean issue loop matters: at N = 128 an MMA lasts ~64 cycles, and
        // rebuilding descriptors per MMA made issue, not the tensor core, the
        // bottleneck.
        constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false);
        constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, kHD, true);
        const uint32_t sbase = smem_addr(smem);
        const uint64_t dQ = umma_desc_sw128(sbase + kOffQ, 16, 1024);    // Q_x: + x * kTileBytes
        const uint64_t dK = umma_desc_sw128(sbase + kOffK, 16, kGroup);    // K stage s: + s * kTileBytes
        const uint64_t dV = umma_desc_sw128(sbase + kOffV, 1024, kGroup);  // V stage s: + s * kTileBytes
        constexpr uint64_t kTileStep = kTileBytes >> 4;
        auto issue_s = [&](int x, int g) {  // S_x = Q_x K_g^T
            if (elect_one()) {
                const uint64_t q = dQ + x * kTileStep, kd = dK + (g % kKStages) * kTileStep;
                const uint32_t d = tmem + x * 128;
#pragma unroll
                for (int k = 0; k < kHD / 16; ++k)  // k-step: 16 columns, 32 B inside the 128-byte atom
                    tc_mma_f16(d, q + (uint64_t)(((k >> 2) * kPanel + (k & 3) * 32) >> 4),
                               kd + (uint64_t)(((k >> 2) * 1024 + (k & 3) * 32) >> 4), idesc_s, k > 0);
                tc_commit(&B.s_full[x]);
            }
            __syncwarp();
        };
        // O_x += P_x V_g, P_x in S_x's first 64 columns; the first tile of an
        // item overwrites O_x (its previous item's epilogue read O_x before
        // the softmax signalled this tile's P)
        auto issue_pv = [&](int x, int g, bool first, bool last) {
            if (elect_one()) {
                const uint64_t vd = dV + (g % kVStages) * kTileStep;
                const uint32_t d = tmem + 256 + x * 128, pa = tmem + x * 128;
#pragma unroll
                for (int k = 0; k < kBN / 16; ++k)  // k-step: 16 keys = two 8-key groups
                    tc_mma_f16_ts(d, pa + k * 8, vd + (uint64_t)((k * 2 * kGroup) >> 4), idesc_o, (!first || k > 0));
                if (x == 1) tc_commit(&B.v_empty[g % kVStages]);
                if (last) tc_commit(&B.o_done[x]);
            }
            __syncwarp();
        };
        auto commit = [&](uint64_t* b) {
            if (elect_one()) tc_commit(b);
            __syncwarp();
        };
        auto wait = [&](uint64_t* b, uint32_t parity) { return warp_wait(b, parity, abort_flag, a.status); };
        int g = 0, ii = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int i = item_index(r);
            if (i < 0) break;
            const int n_kv = item_at(i, false).n_kv;
            if (n_kv == 0) continue;
            // order per tile t: PV_A(t) S_A(t+1) PV_B(t) S_B(t+1); S_x(t+1)
            // overwrites S_x's columns after PV_x(t) has read P_x(t) from them
            // (tensor operations of one thread run in issue order)
            if (!(ok = wait(B.q_full, ii & 1) && wait(&B.k_full[g % kKStages], (g / kKStages) & 1))) break;
            ++ii;
            tc_fence_after();
            issue_s(0, g);
            issue_s(1, g);
            commit(&B.k_empty[g % kKStages]);
            if (n_kv == 1) commit(B.q_empty);
            for (int t = 0; t < n_kv; ++t, ++g) {
                const bool last = t + 1 == n_kv;
                const int g1 = g + 1;
                if (!(ok = wait(&B.v_full[g % kVStages], (g / kVStages) & 1) && wait(&B.p_full[0], g & 1))) break;
                tc_fence_after();
                issue_pv(0, g, t == 0, last);
                if (!last) {
                    if (!(ok = wait(&B.k_full[g1 % kKStages], (g1 / kKStages) & 1))) break;
                    tc_fence_after();
                    issue_s(0, g1);
                }
                if (!(ok = wait(&B.p_full[1], g & 1))) break;
                tc_fence_after();
                issue_pv(1, g, t == 0, last);
                if (!last) {
                    issue_s(1, g1);
                    commit(&B.k_empty[g1 % kKStages]);
                    if (t + 2 == n_kv) commit(B.q_empty);  // the item's last S MMA
                }
            }
        }
        // every MMA this warp issued has completed once `drain` flips
        commit(B.drain);
        mbar_wait(B.drain, 0, a.status);
    } else {
        // ============================ softmax / epilogue ============================
        // Warps 2-9 all work on whichever tile's S is due (A(t), B(t), A(t+1),
        // ...): thread (quarter, lane) owns row r = 32 quarter + lane of the
        // tile, warps 2-5 its columns 0..63 (half hf = 0) and warps 6-9 its
        // columns 64..127 (hf = 1), so two warps per scheduler share each tile.
        // The halves of a row (warps w and w + 4: the same TMEM lane quarter,
        // the same scheduler) agree on the row max through shared memory, with
        // a named barrier of that pair per tile; the barrier ANDs the pair's
        // wait results, so a failed wait stops both halves at the same point
        // (the other pairs stop at their next bounded wait).
        const int hf = (warp - 2) >> 2;
        const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
        const int r = quarter * 32 + lane;        // row of the tile
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        float* xchg = reinterpret_cast<float*>(smem + GE::kOffX);  // [2 tile phases][2 halves][128 rows]
        unsigned char* stage = smem + GE::kOffStage + (warp - 2) * 2048;  // this warp's output staging tile
        const float sl2 = a.scale_log2;
        int g = 0, ii = 0;
        bool ok = true;
        for (int rr_ = 0; ok; ++rr_) {
            const int i = item_index(rr_);
            if (i < 0) break;
            const Item it = item_at(i, false);
            if (it.n_kv == 0) continue;
            float m_used[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
            for (int t = 0; ok && t < it.n_kv; ++t, ++g) {
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const uint32_t tS = tmem + lane_base + x * 128 + hf * 64;
                    const uint32_t tO = tmem + lane_base + 256 + x * 128 + hf * (kHD / 2);
                    const int pos_r = it.pos0 + x * kBM + r;  // absolute position of this row
                    const int pos_first = it.pos0 + x * kBM;  // ... of the tile's first row
                    // keys past the end of the sequence: V rows must be zero (stale
                    // cache slots may hold anything, and 0 * NaN is NaN).  Done in
                    // tile A's phase; PV_B(t) is issued after PV_A(t).
                    const bool zero_v = x == 0 && (t + 1) * kBN > it.seq_len;
                    bool good = warp_wait(&B.s_full[x], g & 1, abort_flag, a.status);
                    if (good && zero_v)
                        good = warp_wait(&B.v_full[g % kVStages], (g / kVStages) & 1, abort_flag, a.status);
                    uint32_t sv[64];
                    float hm = -INFINITY;
                    if (good) {
                        tc_fence_after();
                        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                        tmem_ld_wait();
                        // causal mask: keys past this row's position (only tiles
                        // that reach beyond the tile's first row can have any)
                        if (t * kBN + kBN - 1 > pos_first) {
                            const int lim = pos_r - t * kBN - hf * 64;  // last visible column of this half
#pragma unroll
                            for (int e = 0; e < 64; ++e)
                                if (e > lim) sv[e] = __float_as_uint(-INFINITY);
                        }
                        float m4[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            m4[u] = fmaxf(__uint_as_float(sv[2 * u]), __uint_as_float(sv[2 * u + 1]));
#pragma unroll
                        for (int e = 8; e < 64; e += 8)
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                m4[u] = max3(m4[u], __uint_as_float(sv[e + 2 * u]), __uint_as_float(sv[e + 2 * u + 1]));
                        hm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                    }
                    float* slot = xchg + ((2 * g + x) & 1) * 256;
                    slot[hf * 128 + r] = hm;
                    if (!bar_and(1 + quarter, 64, good)) {
                        ok = false;
                        break;
                    }
                    const float m_tile = fmaxf(hm, slot[(1 - hf) * 128 + r]) * sl2;
                    float alpha = 1.f;
                    bool rescale = false;
                    if (m_used[x] == -INFINITY) {
                        m_used[x] = m_tile;
                    } else if (m_tile > m_used[x] + 8.f) {
                        alpha = fast_exp2(m_used[x] - m_tile);
                        m_used[x] = m_tile;
                        rescale = true;
                    }
                    // P = 2^(s*scale*log2e - m) as bf16 into columns 32hf..32hf+31
                    // of S_x (both halves have read their S before the barrier); a
                    // row with no visible key yet subtracts +inf so every p is 0.
                    // Pairs go through packed f32x2 FMAs and adds; the row sum
                    // adds the fp32 p (their bf16 roundings differ by < 2^-9
                    // relative, at random).
                    const float msub = m_used[x] == -INFINITY ? INFINITY : m_used[x];
                    const uint64_t scale2 = pk(sl2, sl2), msub2 = pk(-msub, -msub);
                    uint64_t sum2[2] = {0, 0};
                    uint32_t pw[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const uint64_t xx =
                            ffma2(pk(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), scale2, msub2);
                        const uint64_t pp = pk(fast_exp2(pk_lo(xx)), fast_exp2(pk_hi(xx)));
                        pw[e] = pack_bf16_rn(pk_lo(pp), pk_hi(pp));
                        sum2[e & 1] = fadd2(sum2[e & 1], pp);
                    }
                    tmem_st32(tmem + lane_base + x * 128 + hf * 32, pw);
                    lsum[x] = lsum[x] * alpha + ((pk_lo(sum2[0]) + pk_hi(sum2[0])) + (pk_lo(sum2[1]) + pk_hi(sum2[1])));
                    // O_x (this half's 64 columns): PV_x(t-1) completed before
                    // S_x(t) was reported.  tcgen05.ld/st are warp-collective: the
                    // whole warp rescales if any of its rows must (alpha is 1 for
                    // the others)
                    if (__any_sync(0xffffffffu, rescale && t > 0)) {
#pragma unroll
                        for (int q = 0; q < kHD / 64; ++q) {
                            uint32_t v[32];
                            tmem_ld32(tO + q * 32, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                            tmem_st32(tO + q * 32, v);
                        }
                    }
                    if (zero_v) {
                        if (t * kBN + r >= it.seq_len) {
                            // key r's row of the V stage: this half zeroes its kHD bytes
                            unsigned char* vrow = smem + kOffV + (g % kVStages) * kTileBytes + (r >> 3) * kGroup +
                                                  (r & 7) * 128 + hf * (kHD == 128 ? 1024 : 64);
#pragma unroll
                            for (int ch = 0; ch < kHD / 16; ++ch)
                                *reinterpret_cast<uint4*>(vrow + ch * 16) = make_uint4(0, 0, 0, 0);
                        }
                        fence_async_smem();
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&B.p_full[x]);
                }
            }
            if (!ok) break;
            // epilogue: O / l -> bf16 rows of out, half hf writing columns
            // hf kHD/2 .. (hf + 1) kHD/2 - 1.  The O reads complete before this item's last
            // arrivals are followed by the next item's first P, which is what
            // lets the next item's first P.V overwrite O.
            const bool good = warp_wait(&B.o_done[0], ii & 1, abort_flag, a.status) &&
                              warp_wait(&B.o_done[1], ii & 1, abort_flag, a.status);
            ++ii;
            float* lx = xchg + 512;  // [2 halves][2 tiles][128 rows]
            lx[(hf * 2 + 0) * 128 + r] = lsum[0];
            lx[(hf * 2 + 1) * 128 + r] = lsum[1];
            if (!bar_and(1 + quarter, 64, good)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const float l = lsum[x] + lx[((1 - hf) * 2 + x) * 128 + r];
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const int row = x * kBM + r;  // row of the 256
                const uint32_t tO = tmem + lane_base + 256 + x * 128 + hf * (kHD / 2);
                // this warp's 32 rows all belong to the item: TMA store of a
                // 32-row x 32-column box per chunk from a 64-byte-swizzled
                // staging tile (rows past the item's end belong to other
                // chunks and are never written: plain stores there)
                const bool full = x * kBM + quarter * 32 + 32 <= it.rows;
#pragma unroll
                for (int q = 0; q < kHD / 64; ++q) {
                    uint32_t v[32];
                    tmem_ld32(tO + q * 32, v);
                    tmem_ld_wait();
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack_bf16_rn(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
                    if (full) {
                        // the previous box's source has been read before it is overwritten
                        if (lane == 0) bulk_wait_group_read0();
                        __syncwarp();
#pragma unroll
                        for (int c = 0; c < 4; ++c)  // 16-byte chunk c of row `lane` at chunk c ^ ((lane >> 1) & 3)
                            *reinterpret_cast<uint4*>(stage + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
                                make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&maps.o, hf * (kHD / 2) + q * 32, it.j, it.row0 + x * kBM + quarter * 32, stage);
                            bulk_commit_group();
                        }
                    } else if (row < it.rows) {
                        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.out) +
                                              ((int64_t)(it.row0 + row) * a.hq + it.j) * kHD + hf * (kHD / 2) + q * 32;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            *reinterpret_cast<uint4*>(orow + 8 * c) =
                                make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                    }
                }
            }
            // the lsum exchange area is rewritten by the next epilogue only
            // after the next item's tile barriers, which every thread reaches
            // after its reads here
        }
        if (lane == 0) bulk_wait_group0();  // output stores complete before the CTA exits
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---- host: tensor maps --------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder()
{
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

template <int kHD>
bool make_maps(const PrefillArgs& a, Maps& m)
{
    EncodeTiled enc = encoder();
    if (!enc) return false;
    std::memset(&m, 0, sizeof(m));
    const cuuint32_t estr[3] = {1, 1, 1};
    {
        const cuuint64_t dims[3] = {(cuuint64_t)kHD, (cuuint64_t)a.hq, (cuuint64_t)a.total_q};
        const cuuint64_t strides[2] = {(cuuint64_t)kHD * 2, (cuuint64_t)a.hq * kHD * 2};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)kBM};
        if (enc(&m.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
        const cuuint32_t obox[3] = {32, 1, 32};
        if (enc(&m.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.out, dims, strides, obox, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    const int64_t rows = (int64_t)a.num_blocks * a.hkv * a.block_size;
    if constexpr (kHD == 128) {
        return pool_maps(a.k_pool, a.v_pool, rows, false, &m.k, &m.v);
    } else {
        // (64 columns, rows): a box of (64, 16) is one 16-row page, [16 rows][128 B]
        const cuuint64_t pdims[2] = {64, (cuuint64_t)rows};
        const cuuint64_t pstrides[1] = {64 * 2};
        const cuuint32_t pbox[2] = {64, 16};
        const cuuint32_t pestr[2] = {1, 1};
        for (int i = 0; i < 2; ++i)
            if (enc(i ? &m.v : &m.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(i ? a.v_pool : a.k_pool),
                    pdims, pstrides, pbox, pestr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return false;
        return true;
    }
}

}  // namespace

bool make_row_maps(const void* k_pool, const void* v_pool, int64_t rows, CUtensorMap* k, CUtensorMap* v)
{
    EncodeTiled enc = encoder();
    if (!enc || rows <= 0) return false;
    // (128 columns, rows): a box of (64, 16) is one 64-column panel of 16 rows
    const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {128 * 2};
    const cuuint32_t box[2] = {64, 16};
    const cuuint32_t estr[2] = {1, 1};
    for (int i = 0; i < 2; ++i)
        if (enc(i ? v : k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(i ? v_pool : k_pool), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    return true;
}

bool make_page_maps(const void* k_pool, const void* v_pool, int64_t rows, CUtensorMap* k, CUtensorMap* v)
{
    EncodeTiled enc = encoder();
    if (!enc || rows <= 0 || rows % 16) return false;
    // (64 columns, 8 rows, 2 panels, rows / 8): a box of (64, 8, 2, 2) is one
    // 16-row page, landing as [8-row group][64-column panel][row][128 B]
    const cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)rows / 8};
    const cuuint64_t strides[3] = {128 * 2, 128, 128 * 2 * 8};
    const cuuint32_t box[4] = {64, 8, 2, 2};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    for (int i = 0; i < 2; ++i)
        if (enc(i ? v : k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(i ? v_pool : k_pool), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    return true;
}

bool pool_maps(const void* k_pool, const void* v_pool, int64_t rows, bool row_boxes, CUtensorMap* k, CUtensorMap* v)
{
    // A caller runs the same cache step after step: the last few encodings
    // of this host thread are kept (a tensor map is a pure function of these
    // arguments).
    struct Entry {
        const void* k_pool;
        const void* v_pool;
        int64_t rows;
        bool row_boxes;
        CUtensorMap k, v;
    };
    constexpr int kEntries = 4;
    thread_local Entry cache[kEntries];
    thread_local int filled = 0, next = 0;
    for (int i = 0; i < filled; ++i) {
        const Entry& e = cache[i];
        if (e.k_pool == k_pool && e.v_pool == v_pool && e.rows == rows && e.row_boxes == row_boxes) {
            *k = e.k;
            *v = e.v;
            return true;
        }
    }
    Entry e;
    if (!(row_boxes ? make_row_maps(k_pool, v_pool, rows, &e.k, &e.v) : make_page_maps(k_pool, v_pool, rows, &e.k, &e.v)))
        return false;
    e.k_pool = k_pool;
    e.v_pool = v_pool;
    e.rows = rows;
    e.row_boxes = row_boxes;
    cache[next] = e;
    next = (next + 1) % kEntries;
    filled = filled < kEntries ? filled + 1 : kEntries;
    *k = e.k;
    *v = e.v;
    return true;
}

namespace {

template <int kHD>
kvattn_status launch_prefill_d(const PrefillArgs& a, cudaStream_t s)
{
    if ((int64_t)a.num_blocks * a.hkv * a.block_size >= ((int64_t)1 << 31)) return KVATTN_ERR_UNSUPPORTED;
    Maps maps;
    if (!make_maps<kHD>(a, maps)) return KVATTN_ERR_CUDA;
    constexpr int kSmem = Geo<kHD>::kSmemBytes;
    static SmemLimit limit;
    if (limit.ensure(reinterpret_cast<const void*>(prefill_kernel<kHD>), kSmem) != cudaSuccess) return KVATTN_ERR_CUDA;
    const int n_qt = (a.max_q_len + 2 * kBM - 1) / (2 * kBM);
    const int64_t items = (int64_t)a.num_chunks * n_qt * a.hq;
    if (items <= 0) return KVATTN_OK;
    if (items > 0x7fffffff) return KVATTN_ERR_UNSUPPORTED;
    const int64_t grid = std::min<int64_t>(items, num_sms());  // persistent: one CTA per SM
    return cuda_status(launch_pdl(prefill_kernel<kHD>, dim3((unsigned)grid), dim3(kThreads), kSmem, s, a, maps, n_qt));
}

}  // namespace

kvattn_status launch_prefill(const PrefillArgs& a, cudaStream_t s)
{
    if (a.hq % a.hkv) return KVATTN_ERR_UNSUPPORTED;
    if (a.d == 128) return launch_prefill_d<128>(a, s);
    if (a.d == 64) return launch_prefill_d<64>(a, s);
    return KVATTN_ERR_UNSUPPORTED;
}

}  // namespace kvattn
