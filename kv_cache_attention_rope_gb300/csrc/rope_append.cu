// Fused rotary position embedding + KV-cache append.
//
// "Tokenizer, KV Cache and RoPE" page, section 4: adjacent pairs (x[2i],
// x[2i+1]) of a query/key head vector rotate by m*theta_i, theta_i =
// base^(-2i/D), m = the token position.  "From-scratch AI inference engine"
// page, section 3.2: the new token's K/V go to the cache index equal to that
// same position.  Every q head is rotated (in place, or into a separate dense
// q buffer), every k head rotated into the cache slot and v copied into the
// cache slot, in 16-byte vectors (8 bf16 / 4 fp32 values).  q, k and v are
// rows at any 16-byte-multiple stride, so they can be the three slices of one
// fused QKV projection output ("hand-written LLM inference engine" series,
// chapter 1, section 5.1: GPT-2's merged c_attn layer).  Persistent CTAs stream the tokens through a shared-memory
// ring (rope_append_pipe_kernel); a token too large for two ring stages takes
// the one-CTA-per-token kernel (rope_append_kernel).
//
// Rounding.  A stored element is round-to-nearest-even of the exact rotation
// of the input values.  The angle is reduced exactly: the rotation speed of
// pair i is held as a 64-bit fixed-point count of turns per position
// (round(theta_i / 2pi * 2^64)), so position * speed mod 2^64 is the angle's
// fraction of a turn with no cancellation at large positions.  Each CTA
// computes its token's (cos, sin) of every pair once, in float-float (about
// 44 bits, quadrant and 1/32-turn sector reduction plus short Taylor series),
// into shared memory.  Fast path: the fp32-rounded twiddle, one packed
// multiply and one packed fma per pair, with a rigorous error bound delta =
// 2^-21 (|x0| + |x1|); if both ends of [y - delta, y + delta] round to the
// same bf16 value that value is the correctly rounded result.  Otherwise (a
// fraction of a percent of the elements, mostly results near zero or near a
// rounding boundary) the pair is recomputed in float-float.  fp32 outputs
// always take the float-float path.
#include <algorithm>
#include <mutex>

#include "kvattn_internal.cuh"

namespace kvattn {
namespace {

// Register pairs for the packed f32x2 arithmetic of this file, built and split
// with mov.b64 so that the compiler places the halves without shift/or code.
__device__ __forceinline__ uint64_t pr(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(__float_as_uint(lo)), "r"(__float_as_uint(hi)));
    return r;
}
__device__ __forceinline__ void pr_halves(uint64_t v, uint32_t& lo, uint32_t& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}

// ---------------------------------------------------------- float-float

struct ff {
    float hi, lo;
};

__device__ __forceinline__ ff two_sum(float a, float b)
{
    float s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

__device__ __forceinline__ ff fast_two_sum(float a, float b)  // needs |a| >= |b| or a == 0
{
    float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ ff two_prod(float a, float b)
{
    float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ ff ff_mul(ff x, ff y)
{
    ff p = two_prod(x.hi, y.hi);
    float t = __fmaf_rn(x.hi, y.lo, __fmul_rn(x.lo, y.hi));
    return fast_two_sum(p.hi, __fadd_rn(p.lo, t));
}

__device__ __forceinline__ ff ff_mul_f(ff x, float y)
{
    ff p = two_prod(x.hi, y);
    return fast_two_sum(p.hi, __fmaf_rn(x.lo, y, p.lo));
}

__device__ __forceinline__ ff ff_add(ff x, ff y)
{
    ff s = two_sum(x.hi, y.hi);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}

__device__ __forceinline__ ff ff_add_f(ff x, float y)
{
    ff s = two_sum(x.hi, y);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}

__device__ __forceinline__ ff ff_neg(ff x) { return {-x.hi, -x.lo}; }

// 2*pi split into float + float (the tail is 2*pi - float(2*pi)).
constexpr float kTwoPiHi = 6.28318548202514648f;
constexpr float kTwoPiLo = -1.7484555314695172e-07f;

// 1/n! split into float + float (host-side double rounding of exact rationals).
struct ffc {
    float hi, lo;
};
__host__ __device__ constexpr ffc make_ffc(double d) { return {(float)d, (float)(d - (double)(float)d)}; }

// Accurate (cos, sin) of the angle u * 2^-64 turns.
// Quadrant reduction (exact swap/negate), then the nearest 1/32 turn k*pi/16
// with |k| <= 4 from a 5-entry float-float table of nested-radical values,
// then Taylor series of the remainder x (|x| <= pi/32): terms above ~1e-6 in
// float-float, the rest in float.  Absolute error about 2^-44.
__device__ __forceinline__ void twiddle_core(uint64_t u, const float4* sector, ff& c_out, ff& s_out)
{
    const uint32_t quad = (uint32_t)((u + (1ull << 61)) >> 62);  // nearest quarter turn
    const int64_t rs = (int64_t)(u - ((uint64_t)quad << 62));     // [-2^61, 2^61)
    const int32_t k = (int32_t)((rs + (1ll << 58)) >> 59);        // nearest 1/32 turn, [-4, 4]
    const int64_t r = rs - ((int64_t)k << 59);                    // [-2^58, 2^58]
    const float r_hi = (float)r;
    const float r_lo = (float)(r - (int64_t)r_hi);
    const ff x = ff_mul({r_hi * 0x1p-64f, r_lo * 0x1p-64f}, {kTwoPiHi, kTwoPiLo});
    const ff x2 = ff_mul(x, x);
    const float t = x2.hi;

    constexpr ffc c2 = make_ffc(-1.0 / 2.0), c4 = make_ffc(1.0 / 24.0);
    constexpr ffc s3 = make_ffc(-1.0 / 6.0);
    // cos x = 1 + x2*(-1/2 + x2*(1/24 + x2*(-1/720 + x2/40320)))
    const float ctail = t * (-1.0f / 720.0f + t * (1.0f / 40320.0f));
    ff cpoly = ff_add_f({c4.hi, c4.lo}, ctail);
    cpoly = ff_add(ff{c2.hi, c2.lo}, ff_mul(x2, cpoly));
    const ff cx = ff_add_f(ff_mul(x2, cpoly), 1.0f);
    // sin x = x + x*x2*(-1/6 + x2*(1/120 - x2/5040))
    const float stail = t * (1.0f / 120.0f - t * (1.0f / 5040.0f));
    const ff spoly = ff_add_f({s3.hi, s3.lo}, stail);
    const ff sx = ff_add(x, ff_mul(ff_mul(x, x2), spoly));

    const float4 e = sector[k < 0 ? -k : k];
    const ff ck = {e.x, e.y};
    const ff sk = k < 0 ? ff{-e.z, -e.w} : ff{e.z, e.w};
    // angle a_k + x
    const ff ca = ff_add(ff_mul(ck, cx), ff_neg(ff_mul(sk, sx)));
    const ff sa = ff_add(ff_mul(sk, cx), ff_mul(ck, sx));
    switch (quad & 3u) {
        case 0: c_out = ca; s_out = sa; break;
        case 1: c_out = ff_neg(sa); s_out = ca; break;
        case 2: c_out = ff_neg(ca); s_out = ff_neg(sa); break;
        default: c_out = sa; s_out = ff_neg(ca); break;
    }
}

__device__ __noinline__ void accurate_twiddle(uint64_t u, const float4* sector, ff& c_out, ff& s_out)
{
    twiddle_core(u, sector, c_out, s_out);
}

// Two angles at once: two independent dependency chains in one body, which
// the scheduler interleaves (a lane's two twiddles one after the other were
// the longest step of the ring's producer).
__device__ __noinline__ void accurate_twiddle2(uint64_t u0, uint64_t u1, const float4* sector, ff& c0, ff& s0, ff& c1,
                                               ff& s1)
{
    twiddle_core(u0, sector, c0, s0);
    twiddle_core(u1, sector, c1, s1);
}

// Round-to-nearest-even of the float-float value y to bf16 bits.
__device__ __forceinline__ uint32_t rne_bf16_ff(ff y)
{
    const uint32_t b = __float_as_uint(y.hi);
    if ((b & 0xffffu) == 0x8000u && y.lo != 0.0f) {
        // y.hi sits exactly on a bf16 rounding boundary: the tail decides
        const bool away = (y.lo > 0.0f) == (y.hi > 0.0f);
        return ((b & 0xffff0000u) + (away ? 0x10000u : 0u)) >> 16;
    }
    __nv_bfloat16 h = __float2bfloat16_rn(y.hi);
    return (uint32_t)(*reinterpret_cast<uint16_t*>(&h));
}

// Rotation of one pair by the float-float twiddle (c, s): about 44 bits.
__device__ __forceinline__ void rotate_pair_ff(float x0, float x1, const float4& cs, ff& y0, ff& y1)
{
    const ff c = {cs.x, cs.y}, s = {cs.z, cs.w};
    y0 = ff_add(ff_mul_f(c, x0), ff_neg(ff_mul_f(s, x1)));
    y1 = ff_add(ff_mul_f(s, x0), ff_mul_f(c, x1));
}

// A pair's twiddle as packed operands: y = x0 * (c, s) + x1 * (-s, c) with
// the fp32 roundings of the float-float (c, s); the float-float value itself
// stays in shared memory for the slow path.
struct Twiddle2 {
    uint64_t cs, sc;  // (c, s), (-s, c)
    const float4* ff; // (c_hi, c_lo, s_hi, s_lo)
};

__device__ __forceinline__ Twiddle2 make_twiddle2(const float4* t)
{
    const float4 v = *t;
    Twiddle2 w;
    w.cs = pr(v.x, v.z);
    w.sc = pr(-v.z, v.x);
    w.ff = t;
    return w;
}

// Slow path of rotate_bf16_word, kept out of line (it runs for well under one
// percent of the words and would otherwise bloat every inlined copy), in two
// levels.
// First, split twiddles: each component t (cos or sin, |t| <= 1) as
// t1 + t2 with t1 = t_hi rounded to 16 significant bits and t2 =
// fl((t_hi - t1) + t_lo), so that |t - t1 - t2| < 2^-39 and a bf16 value (8
// significant bits) times t1 is exact in fp32.  Then
//     y0 = fl(fl(x0 c1 - x1 s1) + fl(x0 c2 - fl(x1 s2)))   (y1 alike)
// has error at most 2^-23 |y| + 5.5 * 2^-39 max(|x0|, |x1|): the roundings of
// the two partial sums and of y, and the twiddle tail.  A bound relative to
// |y| decides most of the words that reach this path, by the same test as the
// fast path with delta = 2^-20 |y| + 2^-36 max|x|.  The rest are rounded from
// a float-float rotation.
__device__ __forceinline__ float split_hi16(float hi)
{
    return __uint_as_float((__float_as_uint(hi) + 0x80u) & 0xffffff00u);
}
__device__ __noinline__ uint32_t rotate_bf16_word_slow(float x0, float x1, float4 ff_cs)
{
    const float c1 = split_hi16(ff_cs.x), s1 = split_hi16(ff_cs.z);
    const float c2 = __fadd_rn(__fsub_rn(ff_cs.x, c1), ff_cs.y), s2 = __fadd_rn(__fsub_rn(ff_cs.z, s1), ff_cs.w);
    const float y0 = __fadd_rn(__fmaf_rn(-x1, s1, __fmul_rn(x0, c1)), __fmaf_rn(-x1, s2, __fmul_rn(x0, c2)));
    const float y1 = __fadd_rn(__fmaf_rn(x0, s1, __fmul_rn(x1, c1)), __fmaf_rn(x0, s2, __fmul_rn(x1, c2)));
    const float d = fmaxf(fmaxf(fabsf(x0), fabsf(x1)) * 0x1p-36f, 0x1p-126f);
    const float up = 1.0f + 0x1p-20f, dn = 1.0f - 0x1p-20f;
    const uint32_t hi = pack_bf16_rn(__fmaf_rn(y0, up, copysignf(d, y0)), __fmaf_rn(y1, up, copysignf(d, y1)));
    const uint32_t lo = pack_bf16_rn(__fmaf_rn(y0, dn, -copysignf(d, y0)), __fmaf_rn(y1, dn, -copysignf(d, y1)));
    if (hi == lo) return hi;
    ff z0, z1;
    rotate_pair_ff(x0, x1, ff_cs, z0, z1);
    return rne_bf16_ff(z0) | (rne_bf16_ff(z1) << 16);
}

// Rotates the bf16 pair packed in `w` (low half = even element).
// Fast path: y = fl(fl(x0 (c, s)) + x1 (-s, c)) with the fp32-rounded
// twiddle, one packed multiply and one packed fma.  Its error is at most
// 3 * 2^-24 (|x0| + |x1|): the twiddle's rounding (2^-24 of each term), the
// product's and the fma's roundings (2^-24 of terms bounded by |x0| + |x1|).
// Rounding test: with delta = 2^-21 (|x0| + |x1|) signed like y, fl(y + delta)
// and fl(y - delta) must round to the same bf16 value (their own rounding
// takes at most 2^-24 |y| <= 2^-24 (|x0| + |x1|) off delta, which leaves a
// margin above the error bound); RNE being monotonic, the exact rotation,
// within the bound of y, then rounds to that value.  Otherwise (well under
// one percent of the words, mostly results near zero or near a rounding
// boundary) the slow path decides.
__device__ __forceinline__ uint32_t rotate_bf16_word(uint32_t w, const Twiddle2& tw)
{
    const float x0 = bf16lo(w), x1 = bf16hi(w);
    const uint64_t y = ffma2(pr(x1, x1), tw.sc, fmul2(pr(x0, x0), tw.cs));
    uint32_t y0, y1;
    pr_halves(y, y0, y1);
    const uint32_t dl = __float_as_uint(0x1p-21f * (fabsf(x0) + fabsf(x1)));
    const uint32_t s0 = y0 & 0x80000000u, s1 = y1 & 0x80000000u;
    uint32_t a0, a1, b0, b1;
    pr_halves(fadd2(y, pr(__uint_as_float(dl | s0), __uint_as_float(dl | s1))), a0, a1);
    pr_halves(fadd2(y, pr(__uint_as_float(dl | (s0 ^ 0x80000000u)), __uint_as_float(dl | (s1 ^ 0x80000000u)))), b0,
              b1);
    const uint32_t hi = pack_bf16_rn(__uint_as_float(a0), __uint_as_float(a1));
    if (hi == pack_bf16_rn(__uint_as_float(b0), __uint_as_float(b1))) return hi;
    return rotate_bf16_word_slow(x0, x1, *tw.ff);
}

template <bool kBF16, int kD>
__global__ void __launch_bounds__(128) rope_append_kernel(const __grid_constant__ RopeArgs a)
{
    pdl_wait();
    constexpr int kPairs = kD / 2;
    constexpr int kEPV = kBF16 ? 8 : 4;  // elements per 16-byte vector
    constexpr int kVPH = kD / kEPV;      // vectors per head
    constexpr int kPPV = kEPV / 2;       // pairs per vector
    constexpr int kGroups = 128 / kVPH;  // threads sharing one column slice
    constexpr int kE = kBF16 ? 2 : 4;
    constexpr int kMaxV = 8;             // vectors a thread keeps in flight
    __shared__ float4 tw[kPairs];        // float-float (cos, sin) of every pair at this position
    __shared__ float4 sector[5];

    const int t = blockIdx.x, tid = threadIdx.x;
    // this thread: column slice dv (fixed), heads hg, hg + kGroups, ... of q, k, v
    const int dv = tid % kVPH, hg = tid / kVPH;
    const int nq = (a.hq - hg + kGroups - 1) / kGroups;   // q heads of this thread
    const int nk = (a.hkv - hg + kGroups - 1) / kGroups;  // k (and v) heads of this thread
    const int nv = max(0, nq) + 2 * max(0, nk);
    auto src_of = [&](int i) -> const char* {  // i-th vector of this thread
        if (i < nq) return (const char*)a.q + t * a.q_stride + ((hg + i * kGroups) * kD + dv * kEPV) * kE;
        i -= nq;
        const bool isv = i >= nk;
        const char* row = isv ? (const char*)a.v + t * a.v_stride : (const char*)a.k + t * a.k_stride;
        if (isv) i -= nk;
        return row + ((hg + i * kGroups) * kD + dv * kEPV) * kE;
    };

    // first loads: independent of the position lookups below
    uint4 w[kMaxV];
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
        if (i < nv) w[i] = *reinterpret_cast<const uint4*>(src_of(i));

    const int pos = a.positions[t];
    const int seq = a.seq_ids[t];
    bool ok = pos >= 0 && seq >= 0 && seq < a.num_seqs && pos / a.block_size < a.max_blocks;
    int64_t blk = -1;
    if (ok) {
        blk = a.block_table[(int64_t)seq * a.max_blocks + pos / a.block_size];
        ok = blk >= 0 && blk < a.num_blocks;
    }
    if (!ok) {
        if (tid == 0) record_error(a.status, KVATTN_ERR_BAD_INDEX);
        return;
    }
    const int off = pos % a.block_size;
    if (tid < 5) sector[tid] = a.sector[tid];
    __syncthreads();
    for (int i = tid; i < kPairs; i += 128) {
        ff c, sn;
        accurate_twiddle((uint64_t)(uint32_t)pos * a.turns[i], sector, c, sn);
        tw[i] = make_float4(c.hi, c.lo, sn.hi, sn.lo);
    }
    __syncthreads();
    Twiddle2 tws[kPPV];
#pragma unroll
    for (int p = 0; p < kPPV; ++p) tws[p] = make_twiddle2(&tw[dv * kPPV + p]);

    for (int base = 0; base < nv; base += kMaxV) {
        if (base > 0) {
#pragma unroll
            for (int i = 0; i < kMaxV; ++i)
                if (base + i < nv) w[i] = *reinterpret_cast<const uint4*>(src_of(base + i));
        }
#pragma unroll
        for (int ii = 0; ii < kMaxV; ++ii) {
            const int i = base + ii;
            if (i >= nv) break;
            char* dst;
            bool rot = true;
            if (i < nq) {
                dst = (char*)a.q_out + t * a.q_out_stride + ((hg + i * kGroups) * kD + dv * kEPV) * kE;
            } else {
                int u = i - nq;
                const bool isv = u >= nk;
                if (isv) u -= nk;
                rot = !isv;
                void* pool = isv ? a.v_pool : a.k_pool;
                const int64_t head = hg + u * kGroups;
                dst = (char*)pool + (((blk * a.hkv + head) * a.block_size + off) * kD + (int64_t)dv * kEPV) * kE;
            }
            uint4 x = w[ii];
            if (rot) {
                if constexpr (kBF16) {
                    x.x = rotate_bf16_word(x.x, tws[0]);
                    x.y = rotate_bf16_word(x.y, tws[1]);
                    x.z = rotate_bf16_word(x.z, tws[2]);
                    x.w = rotate_bf16_word(x.w, tws[3]);
                } else {
                    ff z0, z1, z2, z3;
                    rotate_pair_ff(__uint_as_float(x.x), __uint_as_float(x.y), *tws[0].ff, z0, z1);
                    rotate_pair_ff(__uint_as_float(x.z), __uint_as_float(x.w), *tws[1].ff, z2, z3);
                    x = make_uint4(__float_as_uint(z0.hi), __float_as_uint(z1.hi), __float_as_uint(z2.hi),
                                   __float_as_uint(z3.hi));
                }
            }
            *reinterpret_cast<uint4*>(dst) = x;
        }
    }
}

// ----------------------------------------------------- fp8 (e4m3) cache rows
//
// A head row of the rotated k (or of v) is stored as e4m3 codes with one fp32
// scale per (slot, head): amax = max |r| over the row's bf16 values r,
// s = amax / 448 and inv = 448 / amax (both fp32, correctly rounded; 1 and 1
// for an all-zero row), code = e4m3(r * inv) rounded to nearest even with
// saturation at +-448.  Dequantised value: code * s.  The lanes sharing one
// head row (kLanes consecutive lanes, 8 values each) agree on amax with
// shuffles inside their group.  Returns this lane's 8 codes (first value in
// the low byte) and the row's scale.
template <int kLanes>
__device__ __forceinline__ uint2 quant_row_fp8(const uint4& x, float& scale)
{
    const unsigned lane = threadIdx.x & 31u;
    const unsigned gmask = (kLanes == 32 ? 0xffffffffu : ((1u << kLanes) - 1u) << (lane & ~(unsigned)(kLanes - 1)));
    float v[8] = {bf16lo(x.x), bf16hi(x.x), bf16lo(x.y), bf16hi(x.y),
                  bf16lo(x.z), bf16hi(x.z), bf16lo(x.w), bf16hi(x.w)};
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 1; o < kLanes; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, o));
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const __nv_fp8x2_storage_t lo =
            __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(v[4 * h], inv), __fmul_rn(v[4 * h + 1], inv)),
                                     __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi =
            __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(v[4 * h + 2], inv), __fmul_rn(v[4 * h + 3], inv)),
                                     __NV_SATFINITE, __NV_E4M3);
        w[h] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    scale = sc;
    return make_uint2(w[0], w[1]);
}

// This lane's 8 dims (8 * dv ..) of token r's K row into its fp8 page
// (layout: kvattn_internal.cuh, kF8Page); lane dv == 0 writes the scale.
// V goes through append_v_fp8_kernel.
__device__ __forceinline__ void put_k_page_fp8(unsigned char* page, int r, int dv, uint2 kc, float ks)
{
    *reinterpret_cast<uint2*>(page + r * 128 + (((dv >> 1) ^ f8_swz(r)) << 4) + (dv & 1) * 8) = kc;
    if (dv == 0) reinterpret_cast<float*>(page + kF8KsOff)[r] = ks;
}

// V rows of an fp8 append.  The page stores V transposed (dim d's 16 tokens
// in 16 consecutive bytes), so one token alone can only write single bytes,
// 128 scattered partial-sector writes per head row, which made V the most
// expensive part of a prefill chunk's append.  append_v_fp8_kernel groups
// the tokens into runs of consecutive tokens that land in the same page (the
// tokens of a chunk do, 16 at a time).  A CTA takes a window of 16 tokens;
// one warp-wide scan of the window (and the tokens after it that a run may
// reach) gives every run's start, length, slots and cache block.  A CTA is
// one warp for one (window, KV head): many small CTAs keep every SM's memory
// pipe busy and overlap the scans' latency.  Work items are each run of 2 or
// more tokens and all single-token runs of the window together.  Lanes 2e
// and 2e + 1 quantise token e's row (64 dims each, the row's amax agreed
// with one shuffle) exactly as quant_row_fp8 does.  A run's codes go to a
// shared-memory tile [slot][128 B] (16-byte chunks rotated by the slot,
// conflict-free both ways); lane l then reads dims 4l .. 4l+3 of each group
// of 4 slots, transposes the 4x4 bytes with byte permutes, and writes whole
// 16-byte rows for a full page, 4-byte words for complete groups of 4 slots,
// single bytes only at a run's ragged edges.  Single tokens (a decode step's)
// write their bytes directly, 16 tokens per pass of the warp.
constexpr int kVWin = 16;

// Tokens share a page when they have the same sequence and position / 16
// (the block table is per sequence); -1 for a token the append rejects.
__device__ __forceinline__ long long page_id(const RopeArgs& a, int t, int& pos, int& blk)
{
    pos = a.positions[t];
    const int seq = a.seq_ids[t];
    if (pos < 0 || seq < 0 || seq >= a.num_seqs || pos / a.block_size >= a.max_blocks) return -1;
    blk = a.block_table[(int64_t)seq * a.max_blocks + pos / a.block_size];
    if (blk < 0 || blk >= a.num_blocks) return -1;  // recorded by the ring kernel
    return (long long)seq * (((long long)a.max_blocks * a.block_size) / 16) + pos / 16;
}

// codes of 4 values (first in the low byte), e4m3 RN, saturating
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d, float inv)
{
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(a, inv), __fmul_rn(b, inv)), __NV_SATFINITE,
                                                 __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(c, inv), __fmul_rn(d, inv)), __NV_SATFINITE,
                                                 __NV_E4M3);
    return lo | (hi << 16);
}

// Token t's head h row, this lane's half (dims 64 half ..): codes (chunk i =
// 16 dims in w[i]) and the row's scale.  `pair` masks the lanes taking part.
__device__ __forceinline__ void quant_half_row(const RopeArgs& a, int t, int h, int half, unsigned pair, uint4 (&w)[4],
                                               float& scale)
{
    const uint4* src =
        reinterpret_cast<const uint4*>((const char*)a.v + (int64_t)t * a.v_stride + ((int64_t)h * 128 + 64 * half) * 2);
    uint4 x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = src[i];
    float mx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        mx[i] = fmaxf(fmaxf(fmaxf(fabsf(bf16lo(x[i].x)), fabsf(bf16hi(x[i].x))),
                            fmaxf(fabsf(bf16lo(x[i].y)), fabsf(bf16hi(x[i].y)))),
                      fmaxf(fmaxf(fabsf(bf16lo(x[i].z)), fabsf(bf16hi(x[i].z))),
                            fmaxf(fabsf(bf16lo(x[i].w)), fabsf(bf16hi(x[i].w)))));
    float amax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
    amax = fmaxf(amax, __shfl_xor_sync(pair, amax, 1));
    scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 u0 = x[2 * i], u1 = x[2 * i + 1];
        w[i].x = e4m3x4(bf16lo(u0.x), bf16hi(u0.x), bf16lo(u0.y), bf16hi(u0.y), inv);
        w[i].y = e4m3x4(bf16lo(u0.z), bf16hi(u0.z), bf16lo(u0.w), bf16hi(u0.w), inv);
        w[i].z = e4m3x4(bf16lo(u1.x), bf16hi(u1.x), bf16lo(u1.y), bf16hi(u1.y), inv);
        w[i].w = e4m3x4(bf16lo(u1.z), bf16hi(u1.z), bf16lo(u1.w), bf16hi(u1.w), inv);
    }
}

__device__ __forceinline__ unsigned char* fp8_page(const RopeArgs& a, int blk, int h, int pos)
{
    const int ppb = a.block_size / 16;
    return (unsigned char*)a.k_pool + (((int64_t)blk * a.hkv + h) * ppb + (pos % a.block_size) / 16) * kF8Page;
}

__global__ void __launch_bounds__(32, 24) append_v_fp8_kernel(const __grid_constant__ RopeArgs a)
{
    pdl_wait();
    __shared__ __align__(16) unsigned char tile[16 * 128];
    __shared__ float tsc[16];
    const int lane = threadIdx.x;
    const int t0 = blockIdx.x * kVWin, h = blockIdx.y;
    // scan: lane i holds token t0 - 1 + i (the token before the window, the
    // window, and 15 tokens after it: a run starting in the window ends there)
    const int u = t0 - 1 + lane;
    int pos = 0, blk = 0;
    const long long key = (u >= 0 && u < a.num_tokens) ? page_id(a, u, pos, blk) : -2;
    const long long knext = __shfl_down_sync(0xffffffffu, key, 1);
    const unsigned same_next = __ballot_sync(0xffffffffu, lane < 31 && key >= 0 && key == knext);
    const long long kprev = __shfl_up_sync(0xffffffffu, key, 1);
    const unsigned lead = __ballot_sync(0xffffffffu, lane >= 1 && lane <= kVWin && key >= 0 && key != kprev);
    // run starting at lane b: lanes b .. b + n - 1, n = 1 + the set bits of same_next from bit b on (at most 16)
    const int my_n = min(16, __ffs(~(same_next >> lane)));
    const unsigned singles = lead & __ballot_sync(0xffffffffu, my_n == 1);
    const unsigned multis = lead & ~singles;
    const int nm = __popc(multis), items = nm + (singles ? 1 : 0);
    const int e = lane >> 1, half = lane & 1;
    for (int idx = 0; idx < items; ++idx) {
        if (idx < nm) {
            // ---- a run of n >= 2 tokens in one page
            unsigned m = multis;
            for (int k = idx; k > 0; --k) m &= m - 1;
            const int b = __ffs(m) - 1;
            const int n = __shfl_sync(0xffffffffu, my_n, b);
            const int r = __shfl_sync(0xffffffffu, pos, min(b + e, 31)) & 15;  // slot of token e
            const int blk_b = __shfl_sync(0xffffffffu, blk, b), pos_b = __shfl_sync(0xffffffffu, pos, b);
            if (e < n) {
                uint4 w[4];
                float sc;
                quant_half_row(a, t0 - 1 + b + e, h, half, 0xffffffffu >> (32 - 2 * n), w, sc);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<uint4*>(tile + r * 128 + 16 * ((4 * half + i) ^ (r & 7))) = w[i];
                if (half == 0) tsc[r] = sc;
            }
            const uint32_t cov = __reduce_or_sync(0xffffffffu, e < n ? 1u << r : 0u);
            __syncwarp();
            // lane l: dims 4l .. 4l+3 (chunk l / 4 of every slot row, word l % 4)
            const int c = lane >> 2, wo = 4 * (lane & 3);
            uint32_t o[4][4];  // [dim k][slot group j]
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t x[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int rr = 4 * j + q;
                    x[q] = *reinterpret_cast<const uint32_t*>(tile + rr * 128 + 16 * (c ^ (rr & 7)) + wo);
                }
                const uint32_t t01l = __byte_perm(x[0], x[1], 0x5140), t01h = __byte_perm(x[0], x[1], 0x7362);
                const uint32_t t23l = __byte_perm(x[2], x[3], 0x5140), t23h = __byte_perm(x[2], x[3], 0x7362);
                o[0][j] = __byte_perm(t01l, t23l, 0x5410);
                o[1][j] = __byte_perm(t01l, t23l, 0x7632);
                o[2][j] = __byte_perm(t01h, t23h, 0x5410);
                o[3][j] = __byte_perm(t01h, t23h, 0x7632);
            }
            unsigned char* page = fp8_page(a, blk_b, h, pos_b);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                unsigned char* row = page + kF8VOff + 16 * (4 * lane + k);
                if (cov == 0xffffu) {
                    *reinterpret_cast<uint4*>(row) = make_uint4(o[k][0], o[k][1], o[k][2], o[k][3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t q = (cov >> (4 * j)) & 15u;
                        if (q == 15u) {
                            *reinterpret_cast<uint32_t*>(row + 4 * j) = o[k][j];
                        } else if (q) {
#pragma unroll
                            for (int bb = 0; bb < 4; ++bb)
                                if (q >> bb & 1u) row[4 * j + bb] = (unsigned char)(o[k][j] >> (8 * bb));
                        }
                    }
                }
            }
            if (lane < 16 && (cov >> lane & 1u)) reinterpret_cast<float*>(page + kF8VsOff)[lane] = tsc[lane];
            __syncwarp();  // the tile is reused by the next run
        } else {
            // ---- the window's single-token runs, one per lane pair: bytes straight to their pages
            const int ns = __popc(singles);
            unsigned m = singles;
            for (int k = min(e, 16); k > 0; --k) m &= m - 1;
            const int b = m ? __ffs(m) - 1 : 0;
            const int pb = __shfl_sync(0xffffffffu, pos, b), kb = __shfl_sync(0xffffffffu, blk, b);
            if (e < ns) {
                uint4 w[4];
                float sc;
                quant_half_row(a, t0 - 1 + b, h, half, 0xffffffffu >> (32 - 2 * ns), w, sc);
                unsigned char* page = fp8_page(a, kb, h, pb);
                unsigned char* col = page + kF8VOff + 16 * (64 * half) + (pb & 15);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t v4[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int bb = 0; bb < 4; ++bb)
                            col[16 * (16 * i + 4 * q + bb)] = (unsigned char)(v4[q] >> (8 * bb));
                }
                if (half == 0) reinterpret_cast<float*>(page + kF8VsOff)[pb & 15] = sc;
            }
        }
    }
}

// ------------------------------------------------------- pipelined variant
//
// Persistent CTAs, each taking tokens blockIdx.x, blockIdx.x + gridDim.x, ...
// Warp 4 is the producer: per token one lane starts 1-D bulk copies of the
// token's q, k and v rows into a ring stage, and while they fly the warp looks
// up the token's cache slot and computes its float-float twiddles into the
// same stage.  Warps 0-3 rotate from shared memory and write q out (in place
// or to q_out) and k, v to the cache slot.  A token's loads no longer wait for the previous
// token's compute, so a CTA keeps several tokens' bytes in flight.
// Stage layout: [header 16 B][twiddles, kPairs x 16 B][q row][k row][v row].
constexpr int kPipeConsumers = 4;
constexpr int kPipeThreads = (kPipeConsumers + 1) * 32;
constexpr int kPipeMaxStages = 8;

struct PipeHeader {
    long long blk;  // cache block of the token; -1: invalid token (skipped)
    int off;        // slot in the block
    int pad;
};

template <bool kBF16, int kD, bool kFP8>
__global__ void __launch_bounds__(kPipeThreads, 8) rope_append_pipe_kernel(const __grid_constant__ RopeArgs a,
                                                                         const int stages, const int stage_bytes)
{
    pdl_wait();
    constexpr int kPairs = kD / 2;
    constexpr int kEPV = kBF16 ? 8 : 4;  // elements per 16-byte vector
    constexpr int kVPH = kD / kEPV;      // vectors per head
    constexpr int kPPV = kEPV / 2;       // pairs per vector
    constexpr int kGroups = kPipeConsumers * 32 / kVPH;  // consumer threads sharing one column slice
    constexpr int kE = kBF16 ? 2 : 4;
    constexpr int kTwBytes = kPairs * 16;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float4 sector[5];
    __shared__ uint64_t bars[2 * kPipeMaxStages];
    __shared__ int abort_s;
    uint64_t* full = bars;
    uint64_t* empty = bars + kPipeMaxStages;
    volatile int* abort_flag = &abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t qbytes = (uint32_t)a.hq * kD * kE, kbytes = (uint32_t)a.hkv * kD * kE;
    if (tid < 5) sector[tid] = a.sector[tid];
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 33);  // the producer lane's expect-tx arrival + 32 lanes after the header/twiddles
            mbar_init(&empty[s], kPipeConsumers);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kPipeConsumers) {
        // ================================ producer ================================
        const uint64_t policy = l2_evict_first_policy();
        int n = 0;  // tokens started by this CTA
        // the token's cache slot (the same for every lane), looked up one token
        // ahead: position and sequence at the top of the previous token's
        // turn, the block-table entry after its twiddles, so that neither
        // load's latency sits on this token's path
        // (the entry is range-checked where it is used, so that its load is
        // not waited for at the end of the previous token's turn)
        auto lookup = [&](int pos, int seq, int& blk) -> bool {
            const bool ok = pos >= 0 && seq >= 0 && seq < a.num_seqs && pos / a.block_size < a.max_blocks;
            blk = ok ? a.block_table[(int64_t)seq * a.max_blocks + pos / a.block_size] : -1;
            return ok;
        };
        int pos_n = 0, seq_n = 0, blk_n = -1;
        bool ok_n = false;
        if (blockIdx.x < (unsigned)a.num_tokens) {
            pos_n = a.positions[blockIdx.x];
            seq_n = a.seq_ids[blockIdx.x];
            ok_n = lookup(pos_n, seq_n, blk_n);
        }
        for (int t = blockIdx.x; t < a.num_tokens; t += gridDim.x, ++n) {
            const int s = n % stages, use = n / stages;
            unsigned char* st = smem + (size_t)s * stage_bytes;
            const int pos = pos_n;
            const long long blk = blk_n;
            const bool ok = ok_n && blk >= 0 && blk < a.num_blocks;
            const int tn = t + gridDim.x;
            if (tn < a.num_tokens) {
                pos_n = a.positions[tn];
                seq_n = a.seq_ids[tn];
            }
            bool go = true;
            if (lane == 0) {
                go = !*abort_flag;
                if (go && use > 0) go = mbar_wait(&empty[s], (use - 1) & 1, a.status);
                if (!go) {
                    *abort_flag = 1;
                } else {
                    unsigned char* dq = st + 16 + kTwBytes;
                    mbar_arrive_expect_tx(&full[s], qbytes + (kFP8 ? 1 : 2) * kbytes);  // fp8: V has its own kernel
                    bulk_load(dq, (const char*)a.q + t * a.q_stride, qbytes, &full[s], policy);
                    bulk_load(dq + qbytes, (const char*)a.k + t * a.k_stride, kbytes, &full[s], policy);
                    if (!kFP8)
                        bulk_load(dq + qbytes + kbytes, (const char*)a.v + t * a.v_stride, kbytes, &full[s], policy);
                }
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            if (!go) break;
            if (lane == 0) {
                if (!ok) record_error(a.status, KVATTN_ERR_BAD_INDEX);
                PipeHeader* h = reinterpret_cast<PipeHeader*>(st);
                h->blk = ok ? blk : -1;
                h->off = ok ? pos % a.block_size : 0;
            }
            if (ok) {
                float4* tw = reinterpret_cast<float4*>(st + 16);
                if constexpr (kPairs == 64) {
                    ff c0, s0, c1, s1;
                    accurate_twiddle2((uint64_t)(uint32_t)pos * a.turns[lane], (uint64_t)(uint32_t)pos * a.turns[lane + 32],
                                      sector, c0, s0, c1, s1);
                    tw[lane] = make_float4(c0.hi, c0.lo, s0.hi, s0.lo);
                    tw[lane + 32] = make_float4(c1.hi, c1.lo, s1.hi, s1.lo);
                } else {
                    for (int i = lane; i < kPairs; i += 32) {
                        ff c, sn;
                        accurate_twiddle((uint64_t)(uint32_t)pos * a.turns[i], sector, c, sn);
                        tw[i] = make_float4(c.hi, c.lo, sn.hi, sn.lo);
                    }
                }
            }
            if (tn < a.num_tokens) ok_n = lookup(pos_n, seq_n, blk_n);
            mbar_arrive(&full[s]);  // this lane's header/twiddle writes precede the arrival
        }
        // after an abort, let every armed copy land before the CTA can exit
        if (lane == 0 && *abort_flag) {
            const int m = n < stages ? n : stages;
            for (int p = n - m; p < n; ++p) mbar_wait(&full[p % stages], (p / stages) & 1, a.status);
        }
        return;
    }

    // ================================ consumers ================================
    // thread: column slice dv (fixed), heads hg, hg + kGroups, ... of q, k, v
    const int dv = tid % kVPH, hg = tid / kVPH;
    const int nq = max(0, (a.hq - hg + kGroups - 1) / kGroups);   // q heads of this thread
    const int nk = max(0, (a.hkv - hg + kGroups - 1) / kGroups);  // k (and v) heads of this thread
    constexpr int kHeadStep = kGroups * kD * kE;             // bytes between this thread's heads in a row
    const int slice = (hg * kD + dv * kEPV) * kE;             // byte offset of the first vector in a row
    int n = 0;
    for (int t = blockIdx.x; t < a.num_tokens; t += gridDim.x, ++n) {
        const int s = n % stages, use = n / stages;
        const unsigned char* st = smem + (size_t)s * stage_bytes;
        bool ready = !*abort_flag;
        if (ready) ready = mbar_wait(&full[s], use & 1, a.status);
        ready = __all_sync(0xffffffffu, ready);
        if (!ready) {
            if (lane == 0) *abort_flag = 1;
            break;
        }
        const PipeHeader h = *reinterpret_cast<const PipeHeader*>(st);
        if (h.blk >= 0) {
            Twiddle2 tws[kPPV];
#pragma unroll
            for (int p = 0; p < kPPV; ++p) tws[p] = make_twiddle2(reinterpret_cast<const float4*>(st + 16) + dv * kPPV + p);
            const unsigned char* src = st + 16 + kTwBytes + slice;  // this thread's column slice of head hg
            auto rotate16 = [&](uint4 x) -> uint4 {
                if constexpr (kBF16) {
                    x.x = rotate_bf16_word(x.x, tws[0]);
                    x.y = rotate_bf16_word(x.y, tws[1]);
                    x.z = rotate_bf16_word(x.z, tws[2]);
                    x.w = rotate_bf16_word(x.w, tws[3]);
                } else {
                    ff z0, z1, z2, z3;
                    rotate_pair_ff(__uint_as_float(x.x), __uint_as_float(x.y), *tws[0].ff, z0, z1);
                    rotate_pair_ff(__uint_as_float(x.z), __uint_as_float(x.w), *tws[1].ff, z2, z3);
                    x = make_uint4(__float_as_uint(z0.hi), __float_as_uint(z1.hi), __float_as_uint(z2.hi),
                                   __float_as_uint(z3.hi));
                }
                return x;
            };
            // q heads hg, hg + kGroups, ...: rotated into q_out (in place when q_out == q)
            char* qdst = (char*)a.q_out + t * a.q_out_stride + slice;
            for (int i = 0; i < nq; ++i) {
                const uint4 x = *reinterpret_cast<const uint4*>(src + i * kHeadStep);
                *reinterpret_cast<uint4*>(qdst + i * kHeadStep) = rotate16(x);
            }
            // k (rotated) and v (copied) heads into the token's cache slot
            // pool layout [block][kv head][slot][D]: head hg's slot row, this thread's columns
            const unsigned char* ksrc = src + qbytes;
            if constexpr (kFP8) {
                // e4m3 codes and one scale per (slot, head), in the fp8 page of the token
                static_assert(kBF16 && kD == 128, "fp8 cache pages hold D = 128 rows quantised from bf16");
                const int pages = a.block_size / 16;
                const int64_t page0 = ((int64_t)h.blk * a.hkv + hg) * pages + h.off / 16;
                unsigned char* pg = (unsigned char*)a.k_pool + page0 * kF8Page;
                const int64_t step = (int64_t)kGroups * pages * kF8Page;  // kGroups heads further
                for (int u = 0; u < nk; ++u) {
                    const uint4 x = *reinterpret_cast<const uint4*>(ksrc + u * kHeadStep);
                    float ks;
                    const uint2 kc = quant_row_fp8<kVPH>(rotate16(x), ks);
                    put_k_page_fp8(pg + u * step, h.off & 15, dv, kc, ks);
                }
            } else {
                const int64_t slot =
                    (((int64_t)h.blk * a.hkv + hg) * a.block_size + h.off) * (kD * kE) + dv * kEPV * kE;
                const int64_t pool_step = (int64_t)kGroups * a.block_size * (kD * kE);  // kGroups heads further
                char* kdst = (char*)a.k_pool + slot;
                char* vdst = (char*)a.v_pool + slot;
                for (int u = 0; u < nk; ++u) {
                    const uint4 x = *reinterpret_cast<const uint4*>(ksrc + u * kHeadStep);
                    *reinterpret_cast<uint4*>(kdst + u * pool_step) = rotate16(x);
                    *reinterpret_cast<uint4*>(vdst + u * pool_step) =
                        *reinterpret_cast<const uint4*>(ksrc + kbytes + u * kHeadStep);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

}  // namespace

namespace {

// Pipelined launch: two stages of one token each (within 64 KB per CTA), as
// many persistent CTAs as fit on the GPU (aiming at 8 per SM: more resident
// tokens beat a deeper ring per CTA; measured 2 stages x 8 CTAs 51 us, 4 x 4
// 58 us on the mixed step's 8320 tokens), at most one per token.  Returns
// false (nothing launched) when a token's stage is too large for 2 stages.
template <bool kBF16, int kD, bool kFP8>
bool launch_pipe(const RopeArgs& a, cudaStream_t s, cudaError_t& err)
{
    constexpr int kE = kBF16 ? 2 : 4;
    const int64_t stage = 16 + (int64_t)(kD / 2) * 16 + (int64_t)(a.hq + 2 * a.hkv) * kD * kE;
    const int stages = (int)std::min<int64_t>(2, 65536 / stage);
    if (stages < 2) return false;
    const int bytes = stages * (int)stage;
    auto kern = rope_append_pipe_kernel<kBF16, kD, kFP8>;
    static SmemLimit limit;
    err = limit.ensure(reinterpret_cast<const void*>(kern), bytes);
    if (err != cudaSuccess) return true;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPipeThreads, bytes);
    if (err != cudaSuccess) return true;
    const int grid = (int)std::min<int64_t>(a.num_tokens, (int64_t)num_sms() * std::max(1, per_sm));
    err = launch_pdl(kern, dim3(grid), dim3(kPipeThreads), bytes, s, a, stages, (int)stage);
    return true;
}

template <bool kBF16, int kD>
kvattn_status launch_one(const RopeArgs& a, cudaStream_t s)
{
    cudaError_t err = cudaSuccess;
    if (!launch_pipe<kBF16, kD, false>(a, s, err)) {
        err = launch_pdl(rope_append_kernel<kBF16, kD>, dim3(a.num_tokens), dim3(128), 0, s, a);
    }
    return cuda_status(err);
}

}  // namespace

kvattn_status launch_rope_append(const RopeArgs& a, cudaStream_t s)
{
    const bool bf16 = a.dtype == KVATTN_BF16;
    if (bf16 && a.d == 128) return launch_one<true, 128>(a, s);
    if (bf16 && a.d == 64) return launch_one<true, 64>(a, s);
    if (!bf16 && a.d == 128) return launch_one<false, 128>(a, s);
    if (!bf16 && a.d == 64) return launch_one<false, 64>(a, s);
    return KVATTN_ERR_UNSUPPORTED;
}

kvattn_status launch_rope_append_fp8(const RopeArgs& a, cudaStream_t s)
{
    // the ring kernel only: a token whose bf16 q, k, v do not fit two stages is refused
    cudaError_t err = cudaSuccess;
    bool launched = false;
    if (a.dtype == KVATTN_BF16 && a.d == 128) launched = launch_pipe<true, 128, true>(a, s, err);
    if (!launched) return KVATTN_ERR_UNSUPPORTED;
    if (err != cudaSuccess) return KVATTN_ERR_CUDA;
    return cuda_status(launch_pdl(append_v_fp8_kernel, dim3((unsigned)((a.num_tokens + kVWin - 1) / kVWin), (unsigned)a.hkv),
                                  dim3(32), 0, s, a));
}

}  // namespace kvattn
