// Split kernel of the fused metered split-KV decode.  Templates only: each scheme
// instantiates them in its own translation unit (decode_split_<scheme>.cu), so the
// build compiles them in parallel; the log-sum-exp merge is in decode.cu.
//
// One CTA = (KV split, KV head, group of up to NW sequences); warp w owns one
// sequence.  Each warp streams its sequence's 16-token blocks through a
// private ring of shared-memory stages filled by one-dimensional bulk copies
// (cp.async.bulk, completion on an mbarrier).  For the dithered INT8 scheme
// the dither of a block is regenerated once per CTA by all its threads and
// shared by every sequence of the group (the dither is keyed on layer, KV head,
// position and channel, not on the sequence).
//
// Per block and sequence a warp computes, with mma.m16n8k16 (fp16 in, fp32 acc):
//   logits   S[tok, head] = sum_G s_G(tok) * (codes_G . q - xi_hi,G . q - xi_lo,G . q)
//            codes are exact in fp16 and the dither is split into two fp16 pieces,
//            so the logits carry the compressed keys to ~2^-22;
//   Tier A   eps[tok, head] = W[tok, :] . (||q_b|| / sqrt d)  (the norms as fp16 hi+lo,
//            rounded up) [WitCert summary, Theorem 2];
//   output   O^T[ch, head] += (codes - xi)[ch, tok] . (p * s_V)[tok, head].
// The black-box store (bf16 K_hat, V_hat) runs the same products as bf16 MMAs: keys against
// the query (bf16, or fp32 split into three bf16 pieces), values against the weights split
// into bf16 hi + lo.  With value witnesses, S_V = sum e^(l - m) wv_t rides along with Z and
// gives the value meter E_V = S_V / Z after the merge.
// Tier B u = kappa * sqrt(sum_G s_G^2 * sum_{c in G} q_c^2 / (12 d)) [WitCert
// summary, Tier B paragraph] and the online softmax with the two meter
// accumulators S_X = sum e^(l - m) expm1(c_X) run on the CUDA cores.  The TV
// aggregation min(1, (A^2-1)/2) with A = 1 + S_X/Z [WitCert summary,
// improvements list] is applied after the merge.
//
// Launches chain through programmatic dependent launch.  Every kernel waits for its
// predecessor at some point, so a kernel's completion implies that of everything before
// it.  The merge and most writers wait before they let their successor start; the split
// kernel, and the writers of equal appends to a contiguous store, let their successor start
// at once (such a writer waits on its way out).  So when a split kernel starts, its
// preceding write and the merge before that may still run; neither touches what the split
// reads before it waits: the split waits for its predecessor before staging a block the
// preceding write may touch (p.dirty_blk on; for a one-token append that is the final
// block; this also covers the exact pool, the KIVI tail and value-witness rows), before
// writing its partial results (the merge before may still read the scratch), and, with
// block risks on, before its first risk store.  Older blocks, the dither and the queries
// are used without waiting, so the write's and the previous merge's latency overlap the
// decode.  Per-sequence lengths and page tables, which the split reads at once, are set by
// kernels that precede a writer that waits before its successor starts.
#pragma once
#include <atomic>
#include <cfloat>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace witcert {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLog2eUp = 0x1.715478p+0f;          // log2(e) rounded up
// c^4 coefficient of the expm1 series below c = 1/8: 1/24 raised to cover the dropped
// terms, sum_{k>=5} c^(k-4)/k! < 0.042731 on [0, 1/8), so c(1 + c/2 + c^2/6 + a c^3) >= expm1(c)
constexpr float kSeriesC4 = 0.0428f;
constexpr int kXiKHi = 0, kXiKLo = 4096, kXiV = 8192, kXiBytes = 12288;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per barrier wait

template <int SCHEME> struct Lay;
template <> struct Lay<kInt8> : Int8Layout {};
template <> struct Lay<kRtn> : Int8Layout {};
template <> struct Lay<kFp8> : Fp8Layout {};
template <> struct Lay<kKivi> : KiviLayout {};
template <> struct Lay<kBbox> : BboxLayout {};

// Ring stages per warp, and resident CTAs per SM the compiler plans registers for (four-warp
// CTAs: three, at most 170 registers a thread; single-warp CTAs: twelve, at most 168).
template <int NW> struct Stages { static constexpr int value = 2; };
template <int NW> struct MinBlocks { static constexpr int value = NW >= 16 ? 1 : NW == 4 ? 3 : NW == 1 ? 12 : 2; };

// Dither slots: the CTA regenerates the dither XD = NXI - 2 blocks ahead of the block its
// warps consume, so warps may drift up to two blocks apart (one with three slots, which is
// what two 8-warp CTAs per SM leave room for).  CTAs of up to four warps keep two slots and
// regenerate one block ahead (a warp then waits for every warp to finish the block before the
// one it fills, so they drift at most one block apart): the smaller footprint fits more CTAs
// on an SM.
template <int NW> struct XiSlots { static constexpr int value = NW <= 4 ? 2 : NW == 8 ? 3 : 4; };

// A ring stage holds one block and, behind it, the block's value witnesses.
template <int NW, int SCHEME> struct Smem {
  static constexpr int NST = Stages<NW>::value;
  static constexpr int NXI = SCHEME == kInt8 ? XiSlots<NW>::value : 0;
  static constexpr int NXI_DIV = NXI > 0 ? NXI : 1;      // slot arithmetic (used only when NXI > 0)
  static constexpr int XD = NXI > 2 ? NXI - 2 : 1;
  static constexpr int STB = Lay<SCHEME>::BYTES + kVwBytes;
  static constexpr int kRing = NW * NST * STB;
  // A single-warp CTA forms its key dither in registers where it uses it (each lane's operand
  // fragment is one item of the generator); its slots hold the value dither only.
  static constexpr bool XREG = SCHEME == kInt8 && NW == 1;
  static constexpr int XSLOT = XREG ? kXiBytes - kXiV : kXiBytes;
  static constexpr int XV = XREG ? 0 : kXiV;            // value dither within a slot
  static constexpr int kXi = NXI * XSLOT;
  static constexpr int kRingOff = 0;
  static constexpr int kXiOff = (kRing + 127) / 128 * 128;
  // NW x NST stage barriers (one warp each), then NXI "dither slot filled" and NXI
  // "dither slot free" barriers (NW arrivals each)
  static constexpr int kBarOff = kXiOff + kXi;
  // KIVI: each lane's eight query quads (16 bytes each at most), read again every block, live in
  // shared memory rather than in registers
  static constexpr int kQOff = (kBarOff + (NW * NST + 2 * NXI) * 8 + 15) / 16 * 16;
  static constexpr int kQBytes = SCHEME == kKivi ? NW * 32 * 8 * 16 : 0;
  static constexpr int kBytes = kQOff + kQBytes;
};

// An upper bound of sqrt(x) at most one unit above the correctly rounded value: the SFU
// root, raised one unit while its square (exact sign from one FMA) is below x; the exactly
// rounded-up root if that is still short.
__device__ __forceinline__ float sqrt_up(float x) {
  float y = sqrt_approx(x);
  if (fmaf(y, y, -x) < 0.0f) y = __uint_as_float(__float_as_uint(y) + 1u);
  if (fmaf(y, y, -x) < 0.0f) y = __fsqrt_ru(x);
  return y;
}

// Packed pairs (two query heads of a lane): fp32x2 arithmetic of sm_100+.
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 ex2x2(float2 v) { return make_float2(ex2(v.x), ex2(v.y)); }
// a - b as one packed FMA, b * (-1) + a: the correctly rounded difference, without negating b first
__device__ __forceinline__ float2 f2sub(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a); }

// ------------------------------------------------------------------ meter arithmetic
// The meter is D = S / Z with S = sum_t w_t expm1(c_t) and Z = sum_t w_t over the weights
// w_t = 2^(l_t - m) of one cell.  Its value must never fall below the exact one, whatever
// the length of the sums and the pattern of their roundings:
//  * the running maximum m (log2 units) is kept integer-valued, so every rescale of the sums
//    is a multiplication by an exact power of two;
//  * a lane adds its per-block terms to Z and S in compensated (hi, lo) pairs, moving the
//    low word into the high one by an error-free two-sum every eight blocks (a relative
//    error of at most 8u + O(n u^2), u = 2^-24, for n non-negative terms, instead of the
//    n u of a plain running sum);
//  * lanes, splits and warps are combined with error-free two-sums, and whenever a sum
//    leaves its (hi, lo) pair it is rounded down (Z) or up (S);
//  * the quotient, the margin and D + D^2/2 are rounded up.
// What remains is the rounding of each token's own term (exponentials, logits, witness
// products, the series), a relative error independent of n that kMeterMargin covers.
constexpr float kMeterMargin = 1.0f + 3.0517578125e-5f;   // 1 + 2^-15
// Absolute allowance for terms the flush-to-zero exponentials drop: a dropped term is below
// 2^-126 while Z >= 1/2, so fewer than 2^17 of them move D by less than 2^-108.
constexpr float kMeterFloor = 0x1p-100f;

// 2^k for an integer-valued k <= 0, or k = -inf: the largest float <= 2^k (pow2_dn) and the
// smallest float >= 2^k (pow2_up, never below 2^-149 for a finite k); both are 2^k itself down
// to 2^-149.
__device__ __forceinline__ float pow2_dn(float k) {
  const int e = (int)fmaxf(k, -160.0f) + 127;              // biased exponent of 2^k
  return e > 0 ? __int_as_float(e << 23) : (e > -23 ? __int_as_float(1 << (e + 22)) : 0.0f);
}
__device__ __forceinline__ float pow2_up(float k) {
  return k == -INFINITY ? 0.0f : fmaxf(pow2_dn(k), 0x1p-149f);
}

// Compensated running sum of non-negative terms in (hi, lo) form, two query heads at once: each
// block's term goes into lo with one add, and every kRenorm blocks an error-free two-sum
// (Knuth's, valid for either order of the operands) moves lo's value into hi and leaves its
// rounding error in lo.  An add's error is at most one unit of lo, which holds at most kRenorm
// terms of the current period plus the last two-sum's error, so the errors of a period stay
// below kRenorm u times its sum and the relative error below kRenorm u + O(n u^2) whatever the
// number of blocks n (u = 2^-24).
constexpr int kRenorm = 8;
__device__ __forceinline__ void renorm2(float2& hi, float2& lo) {
  const float2 s = __fadd2_rn(hi, lo);
  const float2 bb = f2sub(s, hi);
  lo = __fadd2_rn(f2sub(hi, f2sub(s, bb)), f2sub(lo, bb));
  hi = s;
}
// (hi, lo) += (ohi, olo) with an error-free two-sum of the high parts (Knuth).
__device__ __forceinline__ void pair_add(float& hi, float& lo, float ohi, float olo) {
  const float s = hi + ohi;
  const float bb = s - hi;
  const float e = (hi - (s - bb)) + (ohi - bb);
  lo = lo + olo + e;
  hi = s;
}

// p * expm1(c) for c >= 0, with p = 2^d the token's weight and d = l - m in log2 units.  Below
// c = 1/8 the series c (1 + c/2 + c^2/6 + a c^3), whose last coefficient a exceeds 1/24 by
// enough that it never falls below expm1(c); above it the term is formed in the exponent,
// 2^(d + c log2 e) - 2^d (log2 e rounded up), which neither overflows for large c nor loses a
// p that flushed to zero, and cancels at most a factor e^c/(e^c - 1) < 8.6 of precision.
// Tokens past the context arrive with d = -inf and c = 0 and give 0.
__device__ __forceinline__ float2 meter_term2(float2 pe, float2 d, float2 c) {
  float2 poly = __ffma2_rn(c, f2(kSeriesC4), f2(1.0f / 6.0f));
  poly = __ffma2_rn(c, poly, f2(0.5f));
  poly = __ffma2_rn(c, poly, f2(1.0f));
  poly = __fmul2_rn(__fmul2_rn(c, poly), pe);
  const float2 big = f2sub(ex2x2(__ffma2_rn(c, f2(kLog2eUp), d)), pe);
  return make_float2(c.x < 0.125f ? poly.x : big.x, c.y < 0.125f ? poly.y : big.y);
}

// The key dither of k-step kk for lane L = 4g + tq of the block whose first token is at
// position tb: tokens g and g + 8, channels 16kk + 4tq .. 16kk + 4tq + 3, as the lane's QK A
// operand, negated, in fp16 hi and lo pieces.  Registers R0 = (g, ch +0,+1), R1 = (g + 8,
// ch +0,+1), R2 = (g, ch +2,+3), R3 = (g + 8, ch +2,+3).
__device__ __forceinline__ void xi_key_frag(const DecodeArgs& p, int h, int tb, int kk, int L, uint32_t (&hw)[4],
                                            uint32_t (&lw)[4]) {
  const int g = L >> 2, quad = 4 * kk + (L & 3);
  const float4 x0 = neg_dither4_rk(p.rk0, p.rk1, p.layer, h, tb + g, quad, 0);
  const float4 x1 = neg_dither4_rk(p.rk0, p.rk1, p.layer, h, tb + g + 8, quad, 0);
  const float2 v[4] = {make_float2(x0.x, x0.y), make_float2(x1.x, x1.y), make_float2(x0.z, x0.w),
                       make_float2(x1.z, x1.w)};
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    // hi = fp16(-xi), lo = fp16(-xi - hi), two values per conversion
    const __half2 hh = __floats2half2_rn(v[r].x, v[r].y);
    const float2 f = __half22float2(hh);
    hw[r] = h2_bits(hh);
    lw[r] = h2_bits(__floats2half2_rn(v[r].x - f.x, v[r].y - f.y));
  }
}

// Regenerate the dither of block `blk` of KV head h into shared memory, in the
// fragment order of the QK operands (negated, fp16 hi + lo) and of the PV operand
// (negated, fp16): each lane's four A registers are contiguous, so one 16-byte load
// fills an MMA operand.  Items 0..255 fill the QK operands, one (k-step, lane) each, with
// 16-byte stores; items 256..511 fill the PV operand, one (token pair, channel quad) each,
// at offset xv.  VONLY: the value items only (the CTA forms its key dither in registers).
template <bool VONLY>
__device__ __forceinline__ void gen_xi(uint8_t* xb, const DecodeArgs& p, int h, int blk, int nthreads, int xv) {
  const int tb = p.pos0 + blk * kBlk;
  for (int idx = (VONLY ? 256 : 0) + threadIdx.x; idx < 512; idx += nthreads) {
    if (!VONLY && idx < 256) {
      uint32_t hw[4], lw[4];
      xi_key_frag(p, h, tb, idx >> 5, idx & 31, hw, lw);
      *reinterpret_cast<uint4*>(xb + kXiKHi + idx * 16) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(xb + kXiKLo + idx * 16) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    } else {
      // Tokens 2pr, 2pr + 1 (pr = t + 4 hi) of channels 4q .. 4q + 3.  Channel c goes to m-tile
      // c >> 4, lane 4 (c & 7) + t, register ((c >> 3) & 1) + 2 hi.  The item's bits are laid
      // out so that a warp's stores fall on 16 banks.
      const int v = idx - 256;
      const int t = v & 3, hi = (v >> 2) & 1, q = ((v >> 4) & 1) | (((v >> 3) & 1) << 1) | ((v >> 5) << 2);
      const int r0 = 2 * (t + 4 * hi);
      const float4 x0 = neg_dither4_rk(p.rk0, p.rk1, p.layer, h, tb + r0, q, 1);
      const float4 x1 = neg_dither4_rk(p.rk0, p.rk1, p.layer, h, tb + r0 + 1, q, 1);
      const float a0[4] = {x0.x, x0.y, x0.z, x0.w}, a1[4] = {x1.x, x1.y, x1.z, x1.w};
      uint32_t* vb = reinterpret_cast<uint32_t*>(xb + xv);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = 4 * q + e;
        vb[((c >> 4) * 32 + 4 * (c & 7) + t) * 4 + ((c >> 3) & 1) + 2 * hi] = h2_bits(__floats2half2_rn(a0[e], a1[e]));
      }
    }
  }
}

// Load four consecutive elements of an exact key row as fp32.
template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <> __device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <> __device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

// Four consecutive elements kept as loaded (bf16: two registers) until they are needed.
template <typename T> struct Raw4;
template <> struct Raw4<float> {
  float4 v;
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ void zero() { v = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ float4 get() const { return v; }
};
template <> struct Raw4<__nv_bfloat16> {
  uint2 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ void zero() { u = make_uint2(0u, 0u); }
  __device__ __forceinline__ float4 get() const {
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
  }
};

// The loaded bits of a bf16 query quad (two bf16 pairs); a float quad has none.
__device__ __forceinline__ uint2 qraw_bits(const Raw4<__nv_bfloat16>& r) { return r.u; }
__device__ __forceinline__ uint2 qraw_bits(const Raw4<float>&) { return make_uint2(0u, 0u); }

// Exact-key logits of one block (repaired block from the pool, or KIVI's unfinished block).
template <typename KT, bool QLO>
__device__ __forceinline__ void exact_block_logits(const KT* ex, const uint32_t (&qb)[8][2],
                                                   const uint32_t (&qbl)[8][2], int g, int t,
                                                   float (&acc)[4]) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const float4 x0 = load4<KT>(ex + g * kD + 16 * kk + 4 * t);
    const float4 x1 = load4<KT>(ex + (g + 8) * kD + 16 * kk + 4 * t);
    __half a0h, a0l, a1h, a1l, b0h, b0l, b1h, b1l, c0h, c0l, c1h, c1l, d0h, d0l, d1h, d1l;
    split_h(x0.x, a0h, a0l); split_h(x0.y, a1h, a1l); split_h(x0.z, b0h, b0l); split_h(x0.w, b1h, b1l);
    split_h(x1.x, c0h, c0l); split_h(x1.y, c1h, c1l); split_h(x1.z, d0h, d0l); split_h(x1.w, d1h, d1l);
    const uint32_t ah[4] = {pack_h2(a0h, a1h), pack_h2(c0h, c1h), pack_h2(b0h, b1h), pack_h2(d0h, d1h)};
    const uint32_t al[4] = {pack_h2(a0l, a1l), pack_h2(c0l, c1l), pack_h2(b0l, b1l), pack_h2(d0l, d1l)};
    mma16816(acc, ah, qb[kk]);
    mma16816(acc, al, qb[kk]);
    if (QLO) mma16816(acc, ah, qbl[kk]);
  }
}

template <int SCHEME, typename QT, bool METER, bool RISK, bool GATE, bool VW, bool PAGED, int NW>
__global__ void __launch_bounds__(NW * 32, MinBlocks<NW>::value) decode_split_kernel(const DecodeArgs p) {
  using L = Lay<SCHEME>;
  using SM = Smem<NW, SCHEME>;
  constexpr int NST = SM::NST;
  constexpr bool QLO = sizeof(QT) == 4;          // fp32 queries carry an fp16 low piece
  extern __shared__ __align__(128) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y;
  const int i = blockIdx.z * p.seqs_per_cta + warp;
  const bool active = warp < p.seqs_per_cta && i < p.B;
  const int grp = p.grp, j0 = h * grp;
  const int nblk = (p.S + kBlk - 1) / kBlk;
  int b_begin, b_end;
  if (nblk < 65536 && p.n_splits < 65536) {
    b_begin = (int)((unsigned)(split * nblk) / (unsigned)p.n_splits);
    b_end = (int)((unsigned)((split + 1) * nblk) / (unsigned)p.n_splits);
  } else {
    b_begin = (int)(((long long)split * nblk) / p.n_splits);
    b_end = (int)(((long long)(split + 1) * nblk) / p.n_splits);
  }
  const int nb = b_end - b_begin;
  // The warp's own sequence length (sequences of a ragged batch differ; the splits cut the
  // longest one's blocks, so block b holds the same positions for every warp and the dither
  // stays shared) and how many of the split's blocks the sequence has.  Every warp still
  // walks all nb blocks for the dither hand-over.
  __shared__ int s_len[NW];                        // read back once per block: keeps a register free
  const int S_w = (p.seq_len && active) ? p.seq_len[i] : p.S;
  const int nbw = min(nb, max(0, (S_w + kBlk - 1) / kBlk - b_begin));
  if (lane == 0) s_len[warp] = S_w;

  constexpr int STB = SM::STB;
  uint8_t* ring = smem + SM::kRingOff + warp * NST * STB;
  uint8_t* xib = smem + SM::kXiOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBarOff) + warp * NST;
  uint64_t* xfull = reinterpret_cast<uint64_t*>(smem + SM::kBarOff) + NW * NST;
  uint64_t* xfree = xfull + SM::NXI;

  const size_t seq_base = active ? ((size_t)(i * p.Hkv + h) * p.nblk_max) : 0;
  const uint8_t* src = p.blocks + (seq_base + b_begin) * L::BYTES;
  // block m of the split: consecutive in a contiguous store, looked up in the page table of a
  // paged one (the same pages serve every layer)
  auto block_src = [&](const uint8_t* base, int m) -> const uint8_t* {
    if constexpr (PAGED) return base + ((size_t)p.table[(size_t)i * p.nblk_max + b_begin + m] * p.Hkv + h) * L::BYTES;
    else return base + (seq_base + b_begin + m) * L::BYTES;
  };
  // one stage: the block (from g) and (value witnesses on) its 32 bytes of value witnesses
  auto stage_copy_from = [&](int s, int m, const uint8_t* g) {
    mbar_expect_tx(smem_addr(&bars[s]), L::BYTES + (VW ? kVwBytes : 0));
    bulk_g2s(smem_addr(ring + s * STB), g, L::BYTES, smem_addr(&bars[s]));
    if (VW)
      bulk_g2s(smem_addr(ring + s * STB + L::BYTES), p.vwit + (seq_base + b_begin + m) * kBlk, kVwBytes,
               smem_addr(&bars[s]));
  };
  auto stage_copy = [&](int s, int m) {
    stage_copy_from(s, m, PAGED ? block_src(p.blocks, m) : src + (size_t)m * L::BYTES);
  };

  // ---------------------------------------------------------------- prologue
  if (SCHEME == kInt8 && threadIdx.x == 0)
    for (int s = 0; s < SM::NXI; ++s) { mbar_init(smem_addr(&xfull[s]), NW); mbar_init(smem_addr(&xfree[s]), NW); }
  if (active && lane == 0)
    for (int s = 0; s < NST; ++s) mbar_init(smem_addr(&bars[s]), 1);
  if ((active && lane == 0) || (SCHEME == kInt8 && threadIdx.x == 0))
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  pdl_trigger();
  // the first blocks' copies go out before anything else; blocks from p.dirty_blk on may
  // still be written by the immediately preceding kernel
  if (active && lane == 0) {
    for (int s = 0; s < NST && s < nbw; ++s) {
      if (b_begin + s >= p.dirty_blk) pdl_wait();
      stage_copy(s, s);
    }
  }
  __syncwarp();

  // ---------------------------------------------------------------- query fragments
  // lane (g, t) holds channels 16kk + 4t .. 16kk + 4t + 3 (kk = 0..7) of query head g: the B
  // fragments of every k-step, the dims of bands t, t+4, t+8, t+12 and 8 channels of each
  // 32-channel group.  The loads are issued here and consumed after the first block's dither.
  const bool has_q = active && g < grp;
  Raw4<QT> qraw[8];
  Raw4<QT>* qsm = reinterpret_cast<Raw4<QT>*>(smem + SM::kQOff) + warp * 8 * 32;   // KIVI only
  {
    const QT* qr = reinterpret_cast<const QT*>(p.q) + ((size_t)(has_q ? i : 0) * p.Hq + j0 + (has_q ? g : 0)) * kD + 4 * t;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      if (has_q) qraw[kk].load(qr + 16 * kk); else qraw[kk].zero();
    }
  }
  bool fault = false;
  // Dither of block b_begin + m into its slot: wait until every warp is done with the block
  // that used the slot before, write this thread's share, then count the warp in.
  auto produce = [&](int m) {
    const int ps = m % SM::NXI_DIV;
    if (m >= SM::NXI && !mbar_wait(smem_addr(&xfree[ps]), (uint32_t)((m / SM::NXI_DIV - 1) & 1), kWaitLimitNs)) {
      if (!fault && lane == 0) atomicAdd(p.err, 1);
      fault = true;
    }
    gen_xi<SM::XREG>(xib + ps * SM::XSLOT, p, h, b_begin + m, NW * 32, SM::XV);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&xfull[ps]));
  };
  if (SCHEME == kInt8) {
    __syncthreads();                  // the dither barriers exist before any warp arrives
    for (int m = 0; m < SM::XD && m < nb; ++m) produce(m);
  }

  uint32_t qb[8][2], qbl[8][2], qnb[2], qnl[2];
  uint32_t qbf[8][2], qbm[8][2], qbs[8][2];      // black-box store: bf16 query pieces
  float qg2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    float bss[4] = {0.f, 0.f, 0.f, 0.f}, gss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const float4 v4 = qraw[kk].get();
      const float v[4] = {v4.x, v4.y, v4.z, v4.w};
      if constexpr (SCHEME == kKivi) qsm[kk * 32 + lane] = qraw[kk];
      __half hv[4], lv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        split_h(v[e], hv[e], lv[e]);
        bss[kk & 3] = __fmaf_ru(v[e], v[e], bss[kk & 3]);
        gss[kk >> 1] = __fmaf_ru(v[e], v[e], gss[kk >> 1]);
      }
      qb[kk][0] = pack_h2(hv[0], hv[1]); qb[kk][1] = pack_h2(hv[2], hv[3]);
      qbl[kk][0] = pack_h2(lv[0], lv[1]); qbl[kk][1] = pack_h2(lv[2], lv[3]);
    }
    if constexpr (SCHEME == kBbox) {
      // bf16 B fragments: a bf16 query as loaded; an fp32 query as hi + mid + lo bf16 pieces
      // (each difference exact in fp32), which sum to the query exactly
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        if constexpr (QLO) {
          const float4 v4 = qraw[kk].get();
          const float v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2 * hf], v[2 * hf + 1]);
            const float r0 = v[2 * hf] - __low2float(hi), r1 = v[2 * hf + 1] - __high2float(hi);
            const __nv_bfloat162 md = __floats2bfloat162_rn(r0, r1);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(r0 - __low2float(md), r1 - __high2float(md));
            qbf[kk][hf] = bf2_bits(hi); qbm[kk][hf] = bf2_bits(md); qbs[kk][hf] = bf2_bits(lo);
          }
        } else {
          const uint2 u = qraw_bits(qraw[kk]);
          qbf[kk][0] = u.x; qbf[kk][1] = u.y;
        }
      }
    }
    if constexpr (SCHEME == kKivi) {
      // KIVI scales the query per block and channel from qraw; exact blocks rebuild the fragments
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) qb[kk][0] = qb[kk][1] = qbl[kk][0] = qbl[kk][1] = 0u;
    }
    qnb[0] = qnb[1] = qnl[0] = qnl[1] = 0u;
    if (METER) {
      // ||q_b|| / sqrt(d) for bands t, t+4 (k 2t, 2t+1) and t+8, t+12 (k 2t+8, 2t+9), rounded up,
      // as fp16 hi + lo (lo rounded up).  0x1.6a09e8p-4 is 1/sqrt(128) rounded up.  The Tier A
      // meter grows like e^eps, so the norm is kept within one unit of its true value.
      __half bh[4], bl[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float nb_up = __fmul_ru(sqrt_up(bss[m]), 0x1.6a09e8p-4f);
        bh[m] = __float2half_rn(nb_up);
        bl[m] = __float2half_ru(nb_up - __half2float(bh[m]));
      }
      qnb[0] = pack_h2(bh[0], bh[1]); qnb[1] = pack_h2(bh[2], bh[3]);
      qnl[0] = pack_h2(bl[0], bl[1]); qnl[1] = pack_h2(bl[2], bl[3]);
      if (SCHEME == kInt8) {
        // sum_{c in G} q_c^2 / (12 d), rounded up (0x1.555556p-11 is 1/1536 rounded up), for
        // heads 2t and 2t+1 (the logit layout)
#pragma unroll
        for (int G = 0; G < 4; ++G) {
          float v = gss[G];
          v = __fadd_ru(v, __shfl_xor_sync(0xffffffffu, v, 1));
          v = __fadd_ru(v, __shfl_xor_sync(0xffffffffu, v, 2));
          gss[G] = __fmul_ru(v, 0x1.555556p-11f);
        }
#pragma unroll
        for (int G = 0; G < 4; ++G) {
          qg2[0][G] = __shfl_sync(0xffffffffu, gss[G], 8 * t);
          qg2[1][G] = __shfl_sync(0xffffffffu, gss[G], 8 * t + 4);
        }
      }
    }
  }
  if (RISK) pdl_wait();    // block risks overwrite rows the preceding merge may still read

  // ---------------------------------------------------------------- state
  // per lane: heads 2t (.x) and 2t+1 (.y); A = token g, B = token g+8 of the block.  m2 is
  // integer-valued; the sums are compensated pairs (hi, lo), renormalized every kRenorm blocks.
  float2 m2 = f2(-INFINITY), Zp = f2(0.f), SAp = f2(0.f), SBp = f2(0.f), SVp = f2(0.f);
  float2 Zl = f2(0.f), SAl = f2(0.f), SBl = f2(0.f), SVl = f2(0.f);
  float acco[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) acco[mt][0] = acco[mt][1] = acco[mt][2] = acco[mt][3] = 0.f;
  float zc[4] = {0.f, 0.f, 0.f, 0.f};           // KIVI: sum_t p_t zero_{t,G} for head g
  const float lscale = kLog2e * 0x1.6a09e6p-4f;   // log2(e) / sqrt(128), 1/sqrt(128) to nearest
  // Tier B: u = kappa * sqrt(var).  var is summed with nearest rounding (4 terms) and the
  // SFU square root is within 2^-22 relative; this factor covers both.
  float kappa = p.kappa;
  if (METER && SCHEME == kInt8 && p.seq_len) {
    // per sequence: sqrt(2 ln(2 S / delta_loc)) in fp64 (log and sqrt within a few units of
    // 2^-53), raised by 2^-40 and rounded up to fp32
    kappa = S_w > 0 ? __double2float_ru(sqrt(2.0 * (log((double)S_w) + p.log2dl)) * (1.0 + 0x1p-40)) : 0.f;
  }
  const float kappa_up = kappa * (1.0f + 1.9073486328125e-6f);
  float2 qgp[4];
#pragma unroll
  for (int G = 0; G < 4; ++G) qgp[G] = make_float2(qg2[0][G], qg2[1][G]);

  const bool gen_early = ((warp >> 2) & 1) == 0;
  // paged store: the page of the block the refill will stage, loaded a block ahead so its
  // latency is off the refill's path
  int32_t page_ahead = 0;
  for (int n = 0; n < nb; ++n) {
    if constexpr (PAGED) {
      if (active && lane == 0 && n + NST < nbw) page_ahead = p.table[(size_t)i * p.nblk_max + b_begin + n + NST];
    }
    const int blk = b_begin + n, stage = n % NST;
    const uint32_t par = (uint32_t)((n / NST) & 1);
    const int xs = SCHEME == kInt8 ? n % SM::NXI_DIV : 0;
    const uint8_t* xb = xib + xs * SM::XSLOT;
    // The dither XD blocks ahead: half of the warps (two per scheduler) make their share before
    // this block's logits, the other half between its softmax and its P.V product, so that the
    // integer work of the one overlaps the tensor and FP32 work of the other.
    const bool gen_next = SCHEME == kInt8 && n + SM::XD < nb;
    if (gen_next && gen_early) produce(n + SM::XD);

    if (active && !fault && n < nbw) {
      if (!mbar_wait(smem_addr(&bars[stage]), par, kWaitLimitNs) ||
          (SCHEME == kInt8 && !mbar_wait(smem_addr(&xfull[xs]), (uint32_t)((n / SM::NXI_DIV) & 1), kWaitLimitNs))) {
        fault = true;
        if (lane == 0) atomicAdd(p.err, 1);
      }
    }
    if (blk >= p.dirty_blk) pdl_wait();             // also covers the exact pool and KIVI tail rows
    const bool live = active && !fault && n < nbw;
    const uint8_t* sb = ring + stage * STB;
    uint32_t P0 = 0u, P1 = 0u, P0l = 0u, P1l = 0u;
    if (live) {
      const int slot = GATE ? p.slots[seq_base + blk] : -1;
      const int S_blk = s_len[warp];
      const bool ragged = (blk + 1) * kBlk > S_blk;    // the context ends inside this block
      const bool kivi_tail = SCHEME == kKivi && ragged;
      float2 lgA, lgB, epsA = f2(0.f), epsB = f2(0.f), ubA = f2(0.f), ubB = f2(0.f);

      if ((GATE && slot >= 0) || kivi_tail) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t fb[8][2], fbl[8][2];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if constexpr (SCHEME == kKivi) {
            const float4 v4 = qsm[kk * 32 + lane].get();
            __half h0, h1, h2, h3, l0, l1, l2, l3;
            split_h(v4.x, h0, l0); split_h(v4.y, h1, l1); split_h(v4.z, h2, l2); split_h(v4.w, h3, l3);
            fb[kk][0] = pack_h2(h0, h1); fb[kk][1] = pack_h2(h2, h3);
            fbl[kk][0] = pack_h2(l0, l1); fbl[kk][1] = pack_h2(l2, l3);
          } else {
            fb[kk][0] = qb[kk][0]; fb[kk][1] = qb[kk][1]; fbl[kk][0] = qbl[kk][0]; fbl[kk][1] = qbl[kk][1];
          }
        }
        if (GATE && slot >= 0)
          exact_block_logits<QT, QLO>(reinterpret_cast<const QT*>(p.pool) + (size_t)slot * kBlk * kD, fb, fbl, g, t, acc);
        else
          exact_block_logits<float, QLO>(p.kivi_tail + seq_base / p.nblk_max * (size_t)(kBlk * kD), fb, fbl, g, t, acc);
        lgA = __fmul2_rn(make_float2(acc[0], acc[1]), f2(lscale));
        lgB = __fmul2_rn(make_float2(acc[2], acc[3]), f2(lscale));
      } else if constexpr (int8_layout(SCHEME)) {
        float acc[4][4];
#pragma unroll
        for (int G = 0; G < 4; ++G) {
          acc[G][0] = acc[G][1] = acc[G][2] = acc[G][3] = 0.f;
          const uint4 cw = *reinterpret_cast<const uint4*>(sb + L::KC + G * 512 + lane * 16);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int kk = 2 * G + hf;
            const uint32_t w0 = hf ? cw.z : cw.x, w1 = hf ? cw.w : cw.y;
            const uint32_t a[4] = {i8x2_lo(w0), i8x2_lo(w1), i8x2_hi(w0), i8x2_hi(w1)};
            mma16816(acc[G], a, qb[kk]);
            if (QLO) mma16816(acc[G], a, qbl[kk]);
            if constexpr (SCHEME != kInt8) continue;                 // no dither to subtract
            uint32_t ah[4], al[4];
            if constexpr (SM::XREG) {
              xi_key_frag(p, h, p.pos0 + blk * kBlk, kk, lane, ah, al);
            } else {
              const uint4 xh = *reinterpret_cast<const uint4*>(xb + kXiKHi + (kk * 32 + lane) * 16);
              const uint4 xl = *reinterpret_cast<const uint4*>(xb + kXiKLo + (kk * 32 + lane) * 16);
              ah[0] = xh.x; ah[1] = xh.y; ah[2] = xh.z; ah[3] = xh.w;
              al[0] = xl.x; al[1] = xl.y; al[2] = xl.z; al[3] = xl.w;
            }
            mma16816(acc[G], ah, qb[kk]);
            mma16816(acc[G], al, qb[kk]);
            if (QLO) mma16816(acc[G], ah, qbl[kk]);
          }
        }
        const __half* ks = reinterpret_cast<const __half*>(sb + L::KS);
        const uint2 s0 = *reinterpret_cast<const uint2*>(ks + g * 4);
        const uint2 s1 = *reinterpret_cast<const uint2*>(ks + (g + 8) * 4);
        const float2 sg01 = __half22float2(bits_h2(s0.x)), sg23 = __half22float2(bits_h2(s0.y));
        const float2 sh01 = __half22float2(bits_h2(s1.x)), sh23 = __half22float2(bits_h2(s1.y));
        const float sgA[4] = {sg01.x, sg01.y, sg23.x, sg23.y}, sgB[4] = {sh01.x, sh01.y, sh23.x, sh23.y};
        lgA = f2(0.f);
        lgB = f2(0.f);
#pragma unroll
        for (int G = 0; G < 4; ++G) {
          lgA = __ffma2_rn(f2(sgA[G]), make_float2(acc[G][0], acc[G][1]), lgA);
          lgB = __ffma2_rn(f2(sgB[G]), make_float2(acc[G][2], acc[G][3]), lgB);
        }
        lgA = __fmul2_rn(lgA, f2(lscale));
        lgB = __fmul2_rn(lgB, f2(lscale));
        if (METER && SCHEME == kInt8) {
          // squares of fp16 scales are exact in fp32
          float2 varA = f2(0.f), varB = f2(0.f);
#pragma unroll
          for (int G = 0; G < 4; ++G) {
            varA = __ffma2_rn(f2(sgA[G] * sgA[G]), qgp[G], varA);
            varB = __ffma2_rn(f2(sgB[G] * sgB[G]), qgp[G], varB);
          }
          ubA = __fmul2_rn(make_float2(sqrt_approx(varA.x), sqrt_approx(varA.y)), f2(kappa_up));
          ubB = __fmul2_rn(make_float2(sqrt_approx(varB.x), sqrt_approx(varB.y)), f2(kappa_up));
        }
      } else if constexpr (SCHEME == kFp8) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};   // two chains
#pragma unroll
        for (int G = 0; G < 4; ++G) {
          const uint4 cw = *reinterpret_cast<const uint4*>(sb + L::KC + G * 512 + lane * 16);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int kk = 2 * G + hf;
            const uint32_t w0 = hf ? cw.z : cw.x, w1 = hf ? cw.w : cw.y;
            const uint32_t a[4] = {e4m3x2_lo(w0), e4m3x2_lo(w1), e4m3x2_hi(w0), e4m3x2_hi(w1)};
            mma16816(hf ? acc2 : acc, a, qb[kk]);
            if (QLO) mma16816(hf ? acc2 : acc, a, qbl[kk]);
          }
        }
        lgA = __fmul2_rn(make_float2(acc[0] + acc2[0], acc[1] + acc2[1]), f2(lscale));
        lgB = __fmul2_rn(make_float2(acc[2] + acc2[2], acc[3] + acc2[3]), f2(lscale));
      } else if constexpr (SCHEME == kBbox) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};   // two chains
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint4 kw = *reinterpret_cast<const uint4*>(sb + L::KH + (kk * 32 + lane) * 16);
          const uint32_t a[4] = {kw.x, kw.y, kw.z, kw.w};
          mma16816_bf16((kk & 1) ? acc2 : acc, a, qbf[kk]);
          if (QLO) {
            mma16816_bf16((kk & 1) ? acc2 : acc, a, qbm[kk]);
            mma16816_bf16((kk & 1) ? acc2 : acc, a, qbs[kk]);
          }
        }
        lgA = __fmul2_rn(make_float2(acc[0] + acc2[0], acc[1] + acc2[1]), f2(lscale));
        lgB = __fmul2_rn(make_float2(acc[2] + acc2[2], acc[3] + acc2[3]), f2(lscale));
      } else {  // KIVI: logits = q . zero + (q * scale) . codes
        // this lane's channels 16kk + 4t + e: their scales (and zeros) are 64 contiguous bytes
        const uint4* sp = reinterpret_cast<const uint4*>(sb + L::KP) + 4 * t;
        const uint4* zp = reinterpret_cast<const uint4*>(sb + L::KP + 256) + 4 * t;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};     // two chains
        float2 zq2 = f2(0.f);
        const uint4 cw = *reinterpret_cast<const uint4*>(sb + L::KC + lane * 16);
        const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const uint4 s4 = sp[kq], z4 = zp[kq];                   // k-steps 2kq and 2kq + 1
          const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w}, zw[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int kk = 2 * kq + hf;
            const float4 q4 = qsm[kk * 32 + lane].get();
            const float2 q01 = make_float2(q4.x, q4.y), q23 = make_float2(q4.z, q4.w);
            zq2 = __ffma2_rn(q01, __half22float2(bits_h2(zw[2 * hf])), zq2);
            zq2 = __ffma2_rn(q23, __half22float2(bits_h2(zw[2 * hf + 1])), zq2);
            // (q * scale) as fp16 hi + lo, two channels per conversion
            const float2 x01 = __fmul2_rn(q01, __half22float2(bits_h2(sw[2 * hf])));
            const float2 x23 = __fmul2_rn(q23, __half22float2(bits_h2(sw[2 * hf + 1])));
            const __half2 h01 = __floats2half2_rn(x01.x, x01.y), h23 = __floats2half2_rn(x23.x, x23.y);
            const float2 r01 = f2sub(x01, __half22float2(h01)), r23 = f2sub(x23, __half22float2(h23));
            const uint32_t bh[2] = {h2_bits(h01), h2_bits(h23)};
            const uint32_t bl[2] = {h2_bits(__floats2half2_rn(r01.x, r01.y)), h2_bits(__floats2half2_rn(r23.x, r23.y))};
            const uint32_t w = words[kk >> 1];
            const int pb = (kk & 1) * 4;
            const uint32_t a[4] = {u2x2(w, pb + 0), u2x2(w, pb + 1), u2x2(w, pb + 2), u2x2(w, pb + 3)};
            mma16816(acc[hf], a, bh);
            mma16816(acc[hf], a, bl);
          }
        }
        float zq = zq2.x + zq2.y;
        zq += __shfl_xor_sync(0xffffffffu, zq, 1);
        zq += __shfl_xor_sync(0xffffffffu, zq, 2);      // lanes 4g..4g+3 hold q_g . zero
        const float zq0 = __shfl_sync(0xffffffffu, zq, 8 * t);
        const float zq1 = __shfl_sync(0xffffffffu, zq, 8 * t + 4);
        lgA = __fmul2_rn(make_float2(acc[0][0] + acc[1][0] + zq0, acc[0][1] + acc[1][1] + zq1), f2(lscale));
        lgB = __fmul2_rn(make_float2(acc[0][2] + acc[1][2] + zq0, acc[0][3] + acc[1][3] + zq1), f2(lscale));
      }

      // Tier A from the stored witness (zero for repaired blocks and KIVI's unfinished block)
      if (METER && !(GATE && slot >= 0)) {
        float eps[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4 wf = *reinterpret_cast<const uint4*>(sb + L::W + lane * 16);
        const uint32_t a[4] = {wf.x, wf.y, wf.z, wf.w};
        mma16816(eps, a, qnb);
        mma16816(eps, a, qnl);
        epsA = make_float2(eps[0], eps[1]);
        epsB = make_float2(eps[2], eps[3]);
      }
      if (GATE && slot >= 0) { ubA = f2(0.f); ubB = f2(0.f); }

      if (ragged) {   // tokens past the context: no weight, no meter term
        const int tok0 = blk * kBlk + g, tok1 = tok0 + 8;
        if (tok0 >= S_blk) { lgA = f2(-INFINITY); epsA = f2(0.f); ubA = f2(0.f); }
        if (tok1 >= S_blk) { lgB = f2(-INFINITY); epsB = f2(0.f); ubB = f2(0.f); }
      }

      // ------------------------------------------------------------ online softmax + meters
      // The running max m2 (an integer in log2 units, at least every logit so far) moves only
      // when a logit of the block exceeds it, to the ceiling of the block's largest logit;
      // otherwise the block's weights are taken against m2 as it stands (p <= 1 either way).
      // A move scales everything accumulated by the power of two 2^(old - new): exact, apart
      // from results below 2^-126, which round down for Z and the output and up for the meter
      // sums.
      float2 dA = f2sub(lgA, m2), dB = f2sub(lgB, m2);
      const bool grows = lgA.x > m2.x || lgA.y > m2.y || lgB.x > m2.x || lgB.y > m2.y;
      if (__any_sync(0xffffffffu, grows)) {
        float2 bm = make_float2(fmaxf(lgA.x, lgB.x), fmaxf(lgA.y, lgB.y));
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          bm.x = fmaxf(bm.x, __shfl_xor_sync(0xffffffffu, bm.x, o));
          bm.y = fmaxf(bm.y, __shfl_xor_sync(0xffffffffu, bm.y, o));
        }
        const float2 mn = make_float2(fmaxf(m2.x, ceilf(bm.x)), fmaxf(m2.y, ceilf(bm.y)));
        // exponent of the move: 0 where m2 stays or where nothing was accumulated yet (the sums
        // are still zero)
        const float kx = (mn.x == m2.x || m2.x == -INFINITY) ? 0.f : m2.x - mn.x;
        const float ky = (mn.y == m2.y || m2.y == -INFINITY) ? 0.f : m2.y - mn.y;
        dA = f2sub(lgA, mn);
        dB = f2sub(lgB, mn);
        m2 = mn;
        // Z and the output take 2^k or, below fp32's range, the next float under it; the S sums
        // the next float above it (never below 2^-149).  The products round to nearest: exact
        // while they stay in fp32's normal range, and off by less than 2^-150 below it, inside
        // the meters' absolute allowance (Z itself, which holds the old maximum's weight, is
        // then at most 2^-83 against the new block's weight of at least 1/2).
        const float2 sc = make_float2(pow2_dn(kx), pow2_dn(ky)), su = make_float2(pow2_up(kx), pow2_up(ky));
        Zp = __fmul2_rn(Zp, sc); Zl = __fmul2_rn(Zl, sc);
        SAp = __fmul2_rn(SAp, su); SAl = __fmul2_rn(SAl, su);
        SBp = __fmul2_rn(SBp, su); SBl = __fmul2_rn(SBl, su);
        if (VW) { SVp = __fmul2_rn(SVp, su); SVl = __fmul2_rn(SVl, su); }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const float2 lo = __fmul2_rn(make_float2(acco[mt][0], acco[mt][1]), sc);
          const float2 hi = __fmul2_rn(make_float2(acco[mt][2], acco[mt][3]), sc);
          acco[mt][0] = lo.x; acco[mt][1] = lo.y; acco[mt][2] = hi.x; acco[mt][3] = hi.y;
        }
        if constexpr (SCHEME == kKivi) {
          // head g's zero accumulator: its factor sits in lane g/2
          const float sa = __shfl_sync(0xffffffffu, sc.x, g >> 1), sbb = __shfl_sync(0xffffffffu, sc.y, g >> 1);
          const float scg = (g & 1) ? sbb : sa;
#pragma unroll
          for (int G = 0; G < 4; ++G) zc[G] *= scg;
        }
      }
      const float2 peA = ex2x2(dA), peB = ex2x2(dB);
      Zl = __fadd2_rn(Zl, __fadd2_rn(peA, peB));
      if (METER) {
        const float2 taA = meter_term2(peA, dA, epsA), taB = meter_term2(peB, dB, epsB);
        SAl = __fadd2_rn(SAl, __fadd2_rn(taA, taB));
        if (VW) {       // value witnesses of tokens g and g + 8 (zero past the context, where p is 0)
          const __half* wv = reinterpret_cast<const __half*>(sb + L::BYTES);
          SVl = __fadd2_rn(SVl, __ffma2_rn(peA, f2(__half2float(wv[g])), __fmul2_rn(peB, f2(__half2float(wv[g + 8])))));
        }
        float2 tbA = f2(0.f), tbB = f2(0.f);
        if (SCHEME == kInt8) {
          tbA = meter_term2(peA, dA, ubA);
          tbB = meter_term2(peB, dB, ubB);
          SBl = __fadd2_rn(SBl, __fadd2_rn(tbA, tbB));
        }
        if (RISK) {
          float2 r = SCHEME == kInt8 ? __fadd2_rn(tbA, tbB) : __fadd2_rn(taA, taB);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            r.x += __shfl_xor_sync(0xffffffffu, r.x, o);
            r.y += __shfl_xor_sync(0xffffffffu, r.y, o);
          }
          if (g == 0) {
            if (2 * t < grp) p.risk_raw[((size_t)i * p.Hq + j0 + 2 * t) * p.nblk_max + blk] = make_float2(m2.x, r.x);
            if (2 * t + 1 < grp) p.risk_raw[((size_t)i * p.Hq + j0 + 2 * t + 1) * p.nblk_max + blk] = make_float2(m2.y, r.y);
          }
        }
      }
      if ((n & (kRenorm - 1)) == kRenorm - 1) {      // warp-uniform
        renorm2(Zp, Zl);
        if (METER) {
          renorm2(SAp, SAl);
          if (SCHEME == kInt8) renorm2(SBp, SBl);
          if (VW) renorm2(SVp, SVl);
        }
      }

      // ------------------------------------------------------------ P V
      // Weights as fp16 (token g / g + 8 by heads 2t, 2t+1), transposed in registers into the
      // B operand: P0 = head g, tokens 2t, 2t+1; P1 = head g, tokens 2t+8, 2t+9.
      if constexpr (SCHEME == kBbox) {
        // bf16 hi + lo of the weights (to 2^-17), each transposed like the fp16 ones
        const __nv_bfloat162 hA = __floats2bfloat162_rn(peA.x, peA.y), hB = __floats2bfloat162_rn(peB.x, peB.y);
        const __nv_bfloat162 lA = __floats2bfloat162_rn(peA.x - __low2float(hA), peA.y - __high2float(hA));
        const __nv_bfloat162 lB = __floats2bfloat162_rn(peB.x - __low2float(hB), peB.y - __high2float(hB));
        P0 = movmatrix_trans(bf2_bits(hA));
        P1 = movmatrix_trans(bf2_bits(hB));
        P0l = movmatrix_trans(bf2_bits(lA));
        P1l = movmatrix_trans(bf2_bits(lB));
      } else {
        P0 = movmatrix_trans(h2_bits(__floats2half2_rn(peA.x, peA.y)));
        P1 = movmatrix_trans(h2_bits(__floats2half2_rn(peB.x, peB.y)));
      }
    }
    if (gen_next && !gen_early) produce(n + SM::XD);
    if (live) {
      if constexpr (SCHEME == kBbox) {
        const uint32_t bh[2] = {P0, P1}, bl[2] = {P0l, P1l};
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const uint4 vw = *reinterpret_cast<const uint4*>(sb + L::VH + (mt * 32 + lane) * 16);
          const uint32_t a[4] = {vw.x, vw.y, vw.z, vw.w};
          mma16816_bf16(acco[mt], a, bh);
          mma16816_bf16(acco[mt], a, bl);
        }
      } else if constexpr (SCHEME == kFp8) {
        const uint32_t bfr[2] = {P0, P1};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 vw = *reinterpret_cast<const uint4*>(sb + L::VC + j * 512 + lane * 16);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint32_t w0 = hf ? vw.z : vw.x, w1 = hf ? vw.w : vw.y;
            const uint32_t a[4] = {e4m3x2_lo(w0), e4m3x2_lo(w1), e4m3x2_hi(w0), e4m3x2_hi(w1)};
            mma16816(acco[2 * j + hf], a, bfr);
          }
        }
      } else if constexpr (int8_layout(SCHEME)) {
        // B_j = (p * s_j) in fp16; A = exact codes, then -xi (dithered scheme)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint2 sv = *reinterpret_cast<const uint2*>(sb + L::VS + (j * 16 + 4 * t) * 2);
          const uint32_t bfr[2] = {h2_bits(__hmul2(bits_h2(P0), bits_h2(sv.x))), h2_bits(__hmul2(bits_h2(P1), bits_h2(sv.y)))};
          const uint4 vw = *reinterpret_cast<const uint4*>(sb + L::VC + j * 512 + lane * 16);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int mt = 2 * j + hf;
            const uint32_t w0 = hf ? vw.z : vw.x, w1 = hf ? vw.w : vw.y;
            const uint32_t a[4] = {i8x2_lo(w0), i8x2_lo(w1), i8x2_hi(w0), i8x2_hi(w1)};
            mma16816(acco[mt], a, bfr);
            if constexpr (SCHEME == kInt8) {
              const uint4 xv = *reinterpret_cast<const uint4*>(xb + SM::XV + (mt * 32 + lane) * 16);
              const uint32_t ax[4] = {xv.x, xv.y, xv.z, xv.w};
              mma16816(acco[mt], ax, bfr);
            }
          }
        }
      } else {  // KIVI values: p*scale times codes, plus p*zero per group
        // [tok][G][scale, zero]: 16 bytes per token; this lane's tokens are 2t, 2t+1, 2t+8, 2t+9,
        // and group j's (scale, zero) of token e is word j of row e
        const uint4* vp4 = reinterpret_cast<const uint4*>(sb + L::VP);
        const uint4 r0 = vp4[2 * t], r1 = vp4[2 * t + 1], r2 = vp4[2 * t + 8], r3 = vp4[2 * t + 9];
        const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
        const uint32_t w2[4] = {r2.x, r2.y, r2.z, r2.w}, w3[4] = {r3.x, r3.y, r3.z, r3.w};
        const float2 p01 = __half22float2(bits_h2(P0)), p23 = __half22float2(bits_h2(P1));
        const uint4 vw4 = *reinterpret_cast<const uint4*>(sb + L::VC + lane * 16);
        const uint32_t vwords[4] = {vw4.x, vw4.y, vw4.z, vw4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 sz0 = __half22float2(bits_h2(w0[j])), sz1 = __half22float2(bits_h2(w1[j]));
          const float2 sz2 = __half22float2(bits_h2(w2[j])), sz3 = __half22float2(bits_h2(w3[j]));
          // sum_t p_t zero_{t,j} of head g over the lane's four tokens, then over the four lanes
          float z = fmaf(p01.x, sz0.y, fmaf(p01.y, sz1.y, fmaf(p23.x, sz2.y, p23.y * sz3.y)));
          z += __shfl_xor_sync(0xffffffffu, z, 1);
          z += __shfl_xor_sync(0xffffffffu, z, 2);
          zc[j] += z;
          const float2 ps01 = __fmul2_rn(p01, make_float2(sz0.x, sz1.x)), ps23 = __fmul2_rn(p23, make_float2(sz2.x, sz3.x));
          const uint32_t bfr[2] = {h2_bits(__floats2half2_rn(ps01.x, ps01.y)), h2_bits(__floats2half2_rn(ps23.x, ps23.y))};
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int pb = hf * 4;
            const uint32_t a[4] = {u2x2(vwords[j], pb + 0), u2x2(vwords[j], pb + 1), u2x2(vwords[j], pb + 2),
                                   u2x2(vwords[j], pb + 3)};
            mma16816(acco[2 * j + hf], a, bfr);
          }
        }
      }
      __syncwarp();
      // refill this stage with the block NST ahead
      if (lane == 0 && n + NST < nbw) {
        if (blk + NST >= p.dirty_blk) pdl_wait();
        fence_proxy_async();
        if constexpr (PAGED)
          stage_copy_from(stage, n + NST, p.blocks + ((size_t)page_ahead * p.Hkv + h) * L::BYTES);
        else
          stage_copy(stage, n + NST);
      }
    }
    if (SCHEME == kInt8) {            // this warp is done with the block's dither slot
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&xfree[xs]));
    }
  }

  // Layers are decoded in order: the first blocks this warp will stream in the next layer go
  // to L2 now, so the next decode's pipeline fill overlaps this one's merge and the next write.
  if (p.next_blocks && active && !fault && lane == 0)
    for (int s = 0; s < NST && s < nbw; ++s) prefetch_l2(block_src(p.next_blocks, s), L::BYTES);
  pdl_wait();     // partial results overwrite scratch the preceding merge may still read
  if (fault) {
    // drain copies still in flight before the CTA's shared memory is released
    if (lane == 0)
      for (int s = 0; s < NST; ++s) mbar_wait(smem_addr(&bars[s]), 0, 100000000ull), mbar_wait(smem_addr(&bars[s]), 1, 100000000ull);
    return;
  }
  if (!active) return;

  // ---------------------------------------------------------------- partial state of this split
  // Each lane's pair leaves rounded down (Z) or up (S_A, S_B, S_V); the eight lanes of a head
  // pair then meet through adds rounded the same way (three one-sided roundings), so the record
  // never understates a meter.
  auto lane_sum = [&](float2 hi, float2 lo, bool up) -> float2 {
    float2 v = up ? make_float2(__fadd_ru(hi.x, lo.x), __fadd_ru(hi.y, lo.y))
                  : make_float2(__fadd_rd(hi.x, lo.x), __fadd_rd(hi.y, lo.y));
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      const float ox = __shfl_xor_sync(0xffffffffu, v.x, o), oy = __shfl_xor_sync(0xffffffffu, v.y, o);
      v = up ? make_float2(__fadd_ru(v.x, ox), __fadd_ru(v.y, oy)) : make_float2(__fadd_rd(v.x, ox), __fadd_rd(v.y, oy));
    }
    return v;
  };
  Zp = lane_sum(Zp, Zl, false);
  if (METER) {
    SAp = lane_sum(SAp, SAl, true);
    if (SCHEME == kInt8) SBp = lane_sum(SBp, SBl, true);
    if (VW) SVp = lane_sum(SVp, SVl, true);
  }
  if (SCHEME == kKivi) {
    // add sum_t p_t zero_{t,G} of heads 2t, 2t+1 (held by lanes 4*head)
    float z0[4], z1[4];
#pragma unroll
    for (int G = 0; G < 4; ++G) {
      z0[G] = __shfl_sync(0xffffffffu, zc[G], 8 * t);
      z1[G] = __shfl_sync(0xffffffffu, zc[G], 8 * t + 4);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      acco[mt][0] += z0[mt >> 1]; acco[mt][2] += z0[mt >> 1];
      acco[mt][1] += z1[mt >> 1]; acco[mt][3] += z1[mt >> 1];
    }
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int head = 2 * t + hh;
    if (head >= grp) continue;
    float* rec = p.part + (((size_t)i * p.Hq + j0 + head) * p.n_splits + split) * kPartStride;
    if (g == 0) {
      *reinterpret_cast<float4*>(rec) = hh ? make_float4(m2.y, Zp.y, SAp.y, SBp.y) : make_float4(m2.x, Zp.x, SAp.x, SBp.x);
      *reinterpret_cast<float4*>(rec + 4) = make_float4(hh ? SVp.y : SVp.x, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      rec[kPartAcc + 16 * mt + g] = acco[mt][hh];
      rec[kPartAcc + 16 * mt + g + 8] = acco[mt][2 + hh];
    }
  }
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Dynamic shared memory above 48 KB is opted into once per kernel and device; `done` is
// the calling kernel's own record (one per instantiation of the caller).
template <typename K>
cudaError_t allow_smem(K kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Launches the split kernel, or (occ != nullptr) reports how many of its CTAs fit on an SM.
template <int SCHEME, typename QT, bool METER, bool RISK, bool GATE, bool VW, bool PAGED, int NW>
cudaError_t run_split(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ) {
  using SM = Smem<NW, SCHEME>;
  static std::atomic<uint64_t> smem_done{0};
  static std::atomic<int> resident{0};
  auto k = decode_split_kernel<SCHEME, QT, METER, RISK, GATE, VW, PAGED, NW>;
  cudaError_t e = allow_smem(k, SM::kBytes, smem_done);
  if (e != cudaSuccess) return e;
  if (occ) {
    int n = resident.load(std::memory_order_relaxed);
    if (n <= 0) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, NW * 32, SM::kBytes);
      if (e != cudaSuccess) return e;
      resident.store(n, std::memory_order_relaxed);
    }
    *occ = n;
    return cudaSuccess;
  }
  return launch_pdl(k, grid, dim3(NW * 32), SM::kBytes, st, pdl, a);
}

template <int SCHEME, typename QT, bool METER, bool RISK, bool GATE, bool VW, bool PAGED>
cudaError_t dispatch_nw(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ) {
  switch (a.seqs_per_cta) {
    case 1: return run_split<SCHEME, QT, METER, RISK, GATE, VW, PAGED, 1>(a, grid, st, pdl, occ);
    case 2: return run_split<SCHEME, QT, METER, RISK, GATE, VW, PAGED, 2>(a, grid, st, pdl, occ);
    case 4: return run_split<SCHEME, QT, METER, RISK, GATE, VW, PAGED, 4>(a, grid, st, pdl, occ);
    case 8: return run_split<SCHEME, QT, METER, RISK, GATE, VW, PAGED, 8>(a, grid, st, pdl, occ);
    default:
      // the black-box store's blocks are too large for 16 warps' rings (seqs_per_cta_for caps it at 8)
      if constexpr (SCHEME == kBbox) return cudaErrorInvalidValue;
      else return run_split<SCHEME, QT, METER, RISK, GATE, VW, PAGED, 16>(a, grid, st, pdl, occ);
  }
}

// Instantiated combinations: meters off with and without a gate; meters on without a gate;
// meters on with a gate, which always keeps block risks; each meters-on case with and
// without value witnesses.
template <int SCHEME, typename QT, bool PAGED>
cudaError_t dispatch_combo(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ) {
  const bool gate = a.slots != nullptr, vw = a.vwit != nullptr;
  if (!a.meter) return gate ? dispatch_nw<SCHEME, QT, false, false, true, false, PAGED>(a, grid, st, pdl, occ)
                            : dispatch_nw<SCHEME, QT, false, false, false, false, PAGED>(a, grid, st, pdl, occ);
  if (gate) return vw ? dispatch_nw<SCHEME, QT, true, true, true, true, PAGED>(a, grid, st, pdl, occ)
                      : dispatch_nw<SCHEME, QT, true, true, true, false, PAGED>(a, grid, st, pdl, occ);
  return vw ? dispatch_nw<SCHEME, QT, true, false, false, true, PAGED>(a, grid, st, pdl, occ)
            : dispatch_nw<SCHEME, QT, true, false, false, false, PAGED>(a, grid, st, pdl, occ);
}

// Paged stores are instantiated for bf16 caches only (the runtime rejects fp32 paged caches).
template <int SCHEME, typename QT>
cudaError_t dispatch_qt(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ) {
  if (a.table == nullptr) return dispatch_combo<SCHEME, QT, false>(a, grid, st, pdl, occ);
  if constexpr (sizeof(QT) == 2) return dispatch_combo<SCHEME, QT, true>(a, grid, st, pdl, occ);
  else return cudaErrorInvalidValue;
}

template <int SCHEME>
cudaError_t dispatch_flags(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ = nullptr) {
  return a.is_bf16 ? dispatch_qt<SCHEME, __nv_bfloat16>(a, grid, st, pdl, occ)
                   : dispatch_qt<SCHEME, float>(a, grid, st, pdl, occ);
}

}  // namespace

// Split-kernel launch (occ == nullptr) or resident CTAs per SM (occ != nullptr), one per scheme.
cudaError_t decode_split_int8(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ);
cudaError_t decode_split_rtn(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ);
cudaError_t decode_split_fp8(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ);
cudaError_t decode_split_kivi(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ);
cudaError_t decode_split_bbox(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ);

}  // namespace witcert
