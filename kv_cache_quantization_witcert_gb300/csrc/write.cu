// Write path: quantize appended keys/values into the block store and compute
// the key witness w_{t,b} = ||r_{t,b}|| of 16 bands [WitCert summary, witness
// paragraph and implementation paragraph].
//
// One warp per (sequence, token, KV head); lane l owns channels 4l..4l+3, so a
// 32-channel scale group is 8 lanes and band b (dims 4b..4b+3 and
// 64+4b..64+4b+3) is lanes b and b+16.  The residual is formed in fp64, where
// x - s*(code - xi) is exact, and the band norm is rounded up to fp16 after a
// 2^-48 relative margin, so the stored witness never falls below the true norm.
// KIVI keys are quantized per channel over a 16-token block when the block's
// last token arrives (one warp per (sequence, KV head) walks the blocks in
// order); until then they wait, exact, in a per-(sequence, head) tail buffer.
// The black-box scheme stores a caller's tensor-function outputs K_hat, V_hat as
// bfloat16 and takes the witness against them.  With the value witness on, every
// writer also stores ||v - v_hat|| over the whole row, rounded up to fp16 the same way.
#include <cfloat>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace witcert {

namespace {

constexpr double kWitMargin = 1.0 + 3.552713678800501e-15;   // 1 + 2^-48

template <typename T> __device__ __forceinline__ void load4f(const T* p, float (&x)[4]);
template <> __device__ __forceinline__ void load4f<float>(const float* p, float (&x)[4]) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
template <> __device__ __forceinline__ void load4f<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xFFFF0000u);
  x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xFFFF0000u);
}
template <typename T> __device__ __forceinline__ void store4(T* p, const T* src) {
  if (sizeof(T) == 4) *reinterpret_cast<float4*>(p) = *reinterpret_cast<const float4*>(src);
  else *reinterpret_cast<uint2*>(p) = *reinterpret_cast<const uint2*>(src);
}

// Four consecutive elements of an input row as loaded (bf16: two registers), converted when used.
template <typename T> struct Row4;
template <> struct Row4<float> {
  float4 v;
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ void get(float (&x)[4]) const { x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w; }
};
template <> struct Row4<__nv_bfloat16> {
  uint2 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ void get(float (&x)[4]) const {
    x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xFFFF0000u);
    x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xFFFF0000u);
  }
};
// A lane's share of one token's inputs: K, V and, for the black-box scheme, K_hat, V_hat.
template <typename T> struct TokIn {
  Row4<T> k, v, kh, vh;
  __device__ __forceinline__ void load(const WriteArgs& a, size_t row, int lane, bool hat) {
    const size_t o = row + 4 * lane;
    k.load(reinterpret_cast<const T*>(a.K) + o);
    v.load(reinterpret_cast<const T*>(a.V) + o);
    if (hat) {
      kh.load(reinterpret_cast<const T*>(a.Kh) + o);
      vh.load(reinterpret_cast<const T*>(a.Vh) + o);
    }
  }
};

__device__ __forceinline__ float grp_max8(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  return v;
}
__device__ __forceinline__ float grp_min8(float v) {
  v = fminf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fminf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  v = fminf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  return v;
}

// Witness of token r from the lane's four fp64 residuals; lanes 0..15 store band `lane`.
__device__ __forceinline__ void store_witness(uint8_t* wreg, int r, const double (&res)[4], int lane, bool zero) {
  double ss = res[0] * res[0] + res[1] * res[1] + res[2] * res[2] + res[3] * res[3];
  ss += __shfl_xor_sync(0xffffffffu, ss, 16);
  if (lane < 16) {
    __half w = __float2half_ru(__double2float_ru(sqrt(ss) * kWitMargin));
    if (zero) w = __float2half_rn(0.f);
    *reinterpret_cast<__half*>(wreg + wit_off(r, lane)) = w;
  }
}

// ---------------------------------------------------------------- fp32 double-float witness
// The stored witness is fp16_ru(w * (1 + 2^-48)) of the fp64 band norm.  GB300's FP64 unit is
// too slow to form every norm in fp64, so the norm is formed from the exact residual in
// double-float (pairs of fp32 with error-free sums and products) to about 2^-44, and the fp16
// rounding is taken from that unless an fp16 value lies within the error band of the
// result or the values leave the safe range; then the warp repeats the fp64 computation.
struct Df {
  float hi, lo;
};
__device__ __forceinline__ Df two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ Df fast_two_sum(float a, float b) {      // |a| >= |b| or a == 0
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ Df two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ Df df_add(Df a, Df b) {
  const Df s = two_sum(a.hi, b.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
// Residual t0 + t1 + t2 + t3 (exact fp32 terms) as a double-float; its absolute error is
// below 2^-46 (|t0| + |t1| + |t2| + |t3|).
__device__ __forceinline__ Df residual_df(float t0, float t1, float t2, float t3) {
  const Df a = two_sum(t0, t1);
  const Df b = two_sum(a.hi, t2);
  const Df c = two_sum(b.hi, t3);
  const float e = __fadd_rn(__fadd_rn(a.lo, b.lo), c.lo);
  return fabsf(c.hi) >= fabsf(e) ? fast_two_sum(c.hi, e) : two_sum(c.hi, e);
}
// Smallest fp16 >= hi + lo (lo below one fp32 unit of hi).
__device__ __forceinline__ __half f16_ru_df(float hi, float lo) {
  __half h = __float2half_ru(hi);
  if (__half2float(h) == hi && lo > 0.f) h = __ushort_as_half((unsigned short)(__half_as_ushort(h) + 1));
  return h;
}

// fp16_ru(w (1 + 2^-48)) of w = sqrt(ss), ss a double-float sum of squares whose norm carries
// an absolute error of at most `err` from the residuals and a relative error of at most `arith`
// from the double-float arithmetic.  Returns false when an fp16 value lies within that error
// band (or ss is too small for the band to mean anything): the caller then takes the fp64 path.
__device__ __forceinline__ bool norm_f16_ru(Df ss, float err, float arith, __half& w16) {
  w16 = __float2half_rn(0.f);
  if (!(ss.hi > 0.f)) return !(err > 0.f);      // an exact zero only when the residuals are exact
  // w = sqrt(ss): correctly rounded root, one correction from the exact remainder
  const float y = __fsqrt_rn(ss.hi);
  const float rem = __fmaf_rn(-y, y, ss.hi);
  const Df w = fast_two_sum(y, __fdividef(__fadd_rn(rem, ss.lo), 2.0f * y));
  // z = w (1 + 2^-48)
  const Df z = fast_two_sum(w.hi, __fmaf_rn(w.hi, 0x1p-48f, w.lo));
  w16 = f16_ru_df(z.hi, z.lo);
  const float band = __fadd_ru(arith, __fdiv_ru(__fmul_ru(4.0f, err), w.hi));
  const float up = __fsub_rn(__fsub_rn(__half2float(w16), z.hi), z.lo);         // >= 0
  const unsigned short bits = __half_as_ushort(w16);
  const float down = bits ? __fadd_rn(__fsub_rn(z.hi, __half2float(__ushort_as_half((unsigned short)(bits - 1)))), z.lo)
                          : INFINITY;
  const float lim = __fmul_ru(__fmul_ru(2.0f, band), z.hi);
  return up > lim && down > lim && ss.hi >= 0x1p-90f;
}

// Sum of squares of the lane's four residuals as a double-float; `bad` flags magnitudes
// outside the range where the double-float error bounds hold.
__device__ __forceinline__ Df lane_sumsq(const Df (&res)[4], bool& bad) {
  Df ss = {0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = fabsf(res[e].hi);
    bad |= a > 0x1p60f || (a != 0.f && a < 0x1p-45f);
    Df sq = two_prod(res[e].hi, res[e].hi);
    sq.lo = __fmaf_rn(2.0f * res[e].hi, res[e].lo, sq.lo);
    ss = df_add(ss, sq);
  }
  return ss;
}

// Lanes 0..15 store band `lane` of token r from the lane's four residuals (double-float, with
// absolute error bound `err` summed over them) and its partner lane's (lane ^ 16).  Returns
// false, storing nothing, when the warp must fall back to the fp64 computation.
__device__ __forceinline__ bool store_witness_df(uint8_t* wreg, int r, const Df (&res)[4], float err, int lane,
                                                 bool zero) {
  bool bad = false;
  Df ss = lane_sumsq(res, bad);
  ss = df_add(ss, {__shfl_xor_sync(0xffffffffu, ss.hi, 16), __shfl_xor_sync(0xffffffffu, ss.lo, 16)});
  err = __fadd_ru(err, __shfl_xor_sync(0xffffffffu, err, 16));
  __half w16 = __float2half_rn(0.f);
  if (lane < 16 && !zero) bad |= !norm_f16_ru(ss, err, 0x1p-40f, w16);
  if (__any_sync(0xffffffffu, bad)) return false;
  if (lane < 16) *reinterpret_cast<__half*>(wreg + wit_off(r, lane)) = w16;
  return true;
}

// ---------------------------------------------------------------- fp32 fast path of the witness
// Most bands are decided in plain fp32: from residual estimates rr_e (each within err_e of the
// exact residual, so the band norm is within the sum of the err_e) the norm is bracketed by
// [w_lo, w_hi], widened by 2^-19 for the rounding of the squares, their sums and the square
// root (together below 2^-21), and by 2^-47 more for the stored witness's 2^-48 margin.  When
// both ends round up to the same fp16 value, that value is the stored witness; otherwise (an
// fp16 value inside the bracket, about one band in a thousand) the double-float path decides.
__device__ __forceinline__ bool bracket_f16_ru(float ss, float err, __half& w16) {
  const float w = __fsqrt_rn(ss);
  const float hi = __fmul_ru(__fadd_ru(w, err), 0x1.00002p+0f);       // (1 + 2^-19) above
  const float lo = fmaxf(__fmul_rd(__fsub_rd(w, err), 0x1.ffffcp-1f), 0.0f);
  const __half h_hi = __float2half_ru(hi);
  w16 = h_hi;
  return __half_as_ushort(h_hi) == __half_as_ushort(__float2half_ru(lo));
}
// Band witness (lanes 0..15 store band `lane`) from the lane's fp32 residual estimates and
// their summed error bound; false, storing nothing, when some band of the warp is undecided.
__device__ __forceinline__ bool store_witness_fast(uint8_t* wreg, int r, const float (&rr)[4], float err, int lane,
                                                   bool zero) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) ss = __fmaf_rn(rr[e], rr[e], ss);
  ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 16));
  err = __fadd_ru(err, __shfl_xor_sync(0xffffffffu, err, 16));
  __half w16 = __float2half_rn(0.f);
  const bool ok = lane >= 16 || zero || bracket_f16_ru(ss, err, w16);
  if (!__all_sync(0xffffffffu, ok)) return false;
  if (lane < 16) *reinterpret_cast<__half*>(wreg + wit_off(r, lane)) = zero ? __float2half_rn(0.f) : w16;
  return true;
}
// Value witness of the whole row (lane 0 stores it) by the same rule; the 32-term sum of squares
// stays within the 2^-19 widening.
__device__ __forceinline__ bool store_rownorm_fast(__half* dst, const float (&rr)[4], float err, int lane) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) ss = __fmaf_rn(rr[e], rr[e], ss);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    err = __fadd_ru(err, __shfl_xor_sync(0xffffffffu, err, o));
  }
  __half w16 = __float2half_rn(0.f);
  const bool ok = bracket_f16_ru(ss, err, w16);
  if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
  if (lane == 0) *dst = w16;
  return true;
}
// Error bound of an fp32 residual estimate rr = RN(d + p) formed from d = RN(u - v) (u - v
// exact: the terms' sum has one rounding each) and an exact or rounded-once p: one unit of
// each result, plus an absolute 2^-148 for results below fp32's normal range.
__device__ __forceinline__ float resid_err(float d, float rr) {
  return __fmaf_ru(0x1p-23f, __fadd_ru(fabsf(d), fabsf(rr)), 0x1p-148f);
}

// ---------------------------------------------------------------- quotients
// x / s rounded to nearest from y = RN(1/s): q0 = RN(x y) is within one unit of x / s, the
// remainder x - q0 s is then exact (one FMA), and RN(q0 + r y) is the correctly rounded
// quotient (Markstein's theorem, as in Cornea, Golliver and Markstein, "Correctness proofs
// outline for Newton-Raphson based floating-point divide and square root algorithms", 1999),
// provided no intermediate leaves fp32's normal range.  The writers need the exact quotient
// only where it can move a code: |x / s| >= 2^-25 with s >= 2^-24, far from that range.
__device__ __forceinline__ float div_rn_by(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = __fmaf_rn(-q0, s, x);
  return __fmaf_rn(r, y, q0);
}
// Nearest integer (ties to even) of z, saturated to [-128, 127]: one conversion.
__device__ __forceinline__ int rint_sat_s8(float z) {
  int c;
  asm("cvt.rni.s8.f32 %0, %1;" : "=r"(c) : "f"(z));
  return (int)(signed char)(c & 0xFF);
}
constexpr float kInv127 = 0x1.020408p-7f;          // RN(1/127)
constexpr float kInv3 = 0x1.555556p-2f;            // RN(1/3)

// Value witness: lane 0 stores the norm of the whole row (all 32 lanes' residuals) at *dst,
// by the same rule; false (nothing stored) when the warp must take the fp64 path.
__device__ __forceinline__ bool store_rownorm_df(__half* dst, const Df (&res)[4], float err, int lane) {
  bool bad = false;
  Df ss = lane_sumsq(res, bad);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    ss = df_add(ss, {__shfl_xor_sync(0xffffffffu, ss.hi, o), __shfl_xor_sync(0xffffffffu, ss.lo, o)});
    err = __fadd_ru(err, __shfl_xor_sync(0xffffffffu, err, o));
  }
  __half w16 = __float2half_rn(0.f);
  if (lane == 0) bad |= !norm_f16_ru(ss, err, 0x1p-34f, w16);
  if (__any_sync(0xffffffffu, bad)) return false;
  if (lane == 0) *dst = w16;
  return true;
}
__device__ __forceinline__ void store_rownorm(__half* dst, const double (&res)[4], int lane) {
  double ss = res[0] * res[0] + res[1] * res[1] + res[2] * res[2] + res[3] * res[3];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) *dst = __float2half_ru(__double2float_ru(sqrt(ss) * kWitMargin));
}
// Where token t of (sequence i, KV head h) keeps its value witness.
__device__ __forceinline__ __half* vwit_at(const WriteArgs& a, int i, int h, int t) {
  return a.vwit + (((size_t)i * a.Hkv + h) * a.nblk_max + (t >> 4)) * kBlk + (t & 15);
}

// Entry of a write kernel into the launch chain.  Normally it waits for its predecessor, then
// lets its successor start.  With late_wait (equal appends to a contiguous store) it lets the
// successor start at once, does its work alongside the predecessor (a merge, or a write
// kernel of the same call on other blocks: none of them touches what this kernel touches),
// and waits for the predecessor on its way out, so its completion still implies the
// predecessor's and every later kernel finds all earlier work done.
struct ChainEntry {
  bool late;
  __device__ explicit ChainEntry(bool late_wait) : late(late_wait) {
    if (!late) pdl_wait();
    pdl_trigger();
  }
  __device__ ~ChainEntry() {
    if (late) pdl_wait();
  }
};

// Exact-key side effects shared by all schemes: backing store and repaired blocks.
template <typename T>
__device__ __forceinline__ bool exact_side(const WriteArgs& a, int i, int h, int t, int lane, const T* krow) {
  const size_t sh = (size_t)i * a.Hkv + h;
  if (a.backing) store4<T>(reinterpret_cast<T*>(a.backing) + (sh * a.backing_rows + t) * kD + 4 * lane, krow + 4 * lane);
  if (a.slots) {
    const int slot = a.slots[sh * a.nblk_max + (t >> 4)];
    if (slot >= 0) {
      store4<T>(reinterpret_cast<T*>(a.pool) + ((size_t)slot * kBlk + (t & 15)) * kD + 4 * lane, krow + 4 * lane);
      return true;
    }
  }
  return false;
}

// The token at position t (row r = t mod 16 of its block) of sequence i, KV head h, whose
// input row starts at element `row` of K and V (this lane's part already loaded in `in`),
// quantized into the block image at bp (device memory or shared memory).  STAGED: the value
// codes go, as one word of four channels per lane, to row r of the warp's staging area vst
// (natural order) instead of their places in the block.
template <typename T, bool DITHER, bool VW, bool STAGED>
__device__ __forceinline__ void int8_token(const WriteArgs& a, uint8_t* bp, uint32_t* vst, int i, int h, int t,
                                           size_t row, int lane, const TokIn<T>& in) {
  const int r = t & 15;
  const bool repaired = exact_side<T>(a, i, h, t, lane, reinterpret_cast<const T*>(a.K) + row);
  const int G = lane >> 3;
#pragma unroll
  for (int tensor = 0; tensor < 2; ++tensor) {
    float x[4];
    (tensor ? in.v : in.k).get(x);
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    amax = grp_max8(amax);
    // s = fp16 round-up of fp32(amax / 127), at most 65504
    __half s16 = __float2half_ru(div_rn_by(amax, 127.0f, kInv127));
    if (__half2float(s16) > 65504.0f) s16 = __float2half_rn(65504.0f);
    const float s = __half2float(s16);
    const float ys = s > 0.0f ? __frcp_rn(s) : 0.0f;
    // round to nearest is the dithered quantizer with xi = 0
    const float4 xi = DITHER ? dither4_rk(a.rk0, a.rk1, a.layer, h, a.pos0 + t, lane, tensor)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    const float xs[4] = {xi.x, xi.y, xi.z, xi.w};
    uint32_t packed = 0;
    int codes[4];
    float rr[4], zs[4];
    float eacc = 0.f;
    const bool resid = tensor == 0 || VW;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      // an all-zero group has s = 0 and ys = 0: z = xi, whose nearest integer is 0
      const float z = __fadd_rn(div_rn_by(x[e], s, ys), xs[e]);
      zs[e] = z;
      const int code = rint_sat_s8(z);
      codes[e] = code;
      if (resid) {
        // residual x - s (code - xi) = (x - s code) + s xi: s code is exact (at most 19
        // significant bits), the difference and the FMA round once each, so the estimate is
        // within one unit of |d| and of |rr|
        const float d = __fsub_rn(x[e], __fmul_rn(s, (float)code));
        rr[e] = __fmaf_rn(s, xs[e], d);
        eacc = __fadd_rn(eacc, __fadd_rn(fabsf(d), fabsf(rr[e])));
      }
      const uint32_t biased = (uint32_t)(code ^ 0x80) & 0xFFu;       // code + 128
      if (tensor == 0 || STAGED) packed |= biased << (8 * e);
      else bp[Int8Layout::VC + vcode_off(r, 4 * lane + e)] = (uint8_t)biased;
    }
    // sum of the four one-unit bounds, 2^-24 (|d| + |rr|) each plus 2^-150 below fp32's normal
    // range: the rounded sum eacc is within 2^-21 of exact, so 2^-22 eacc + 2^-146 covers them
    const float ferr = resid ? __fmaf_ru(eacc, 0x1p-22f, 0x1p-146f) : 0.f;
    if (STAGED && tensor == 1) vst[r * 32 + lane] = packed;
    // clamped codes (expected none: s >= amax / 127 keeps |x / s| <= 127 unless s saturated)
    if (fminf(fminf(zs[0], zs[1]), fminf(zs[2], zs[3])) < -128.5f || fmaxf(fmaxf(zs[0], zs[1]), fmaxf(zs[2], zs[3])) >= 127.5f) {
      int clamps = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) clamps += (zs[e] < -128.5f) + (zs[e] >= 127.5f);
      atomicAdd(a.clamps, (unsigned long long)clamps);
    }
    if ((lane & 7) == 0)
      *reinterpret_cast<__half*>(bp + (tensor ? Int8Layout::VS + vscale_off(r, G) : Int8Layout::KS + (r * 4 + G) * 2)) = s16;
    // exact residual terms for the double-float path (x, -s code, and s xi as an exact product pair)
    auto resid_df = [&](Df (&rdf)[4], float& err) {
      err = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float sc = __fmul_rn(s, (float)codes[e]);
        const Df sx = two_prod(s, xs[e]);
        rdf[e] = residual_df(x[e], -sc, sx.hi, sx.lo);
        err = __fadd_ru(err, __fmul_ru(0x1p-46f, __fadd_ru(__fadd_ru(fabsf(x[e]), fabsf(sc)),
                                                           __fadd_ru(fabsf(sx.hi), fabsf(sx.lo)))));
      }
    };
    Df rdf[4];
    float err = 0.f;
    if (tensor == 0) {
      *reinterpret_cast<uint32_t*>(bp + Int8Layout::KC + kcode_off(r, 4 * lane)) = packed;
      if (store_witness_fast(bp + Int8Layout::W, r, rr, ferr, lane, repaired)) continue;
      resid_df(rdf, err);
      if (!store_witness_df(bp + Int8Layout::W, r, rdf, err, lane, repaired)) {
        double res[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) res[e] = (double)x[e] - (double)s * ((double)codes[e] - (double)xs[e]);
        store_witness(bp + Int8Layout::W, r, res, lane, repaired);
      }
    } else if (VW && !store_rownorm_fast(vwit_at(a, i, h, t), rr, ferr, lane)) {
      resid_df(rdf, err);
      if (!store_rownorm_df(vwit_at(a, i, h, t), rdf, err, lane)) {
        double res[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) res[e] = (double)x[e] - (double)s * ((double)codes[e] - (double)xs[e]);
        store_rownorm(vwit_at(a, i, h, t), res, lane);
      }
    }
  }
}

// As int8_token, for the raw FP8 cast.
template <typename T, bool STAGED>
__device__ __forceinline__ void fp8_token(const WriteArgs& a, uint8_t* bp, uint32_t* vst, int i, int h, int t,
                                          size_t row, int lane, const TokIn<T>& in) {
  const int r = t & 15;
  const bool repaired = exact_side<T>(a, i, h, t, lane, reinterpret_cast<const T*>(a.K) + row);
#pragma unroll
  for (int tensor = 0; tensor < 2; ++tensor) {
    float x[4];
    (tensor ? in.v : in.k).get(x);
    uint32_t packed = 0;
    float xhs[4], rr[4];
    Df rdf[4];
    float ferr = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(x[e], __NV_SATFINITE, __NV_E4M3);
      const float xh = __half2float(__half(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3)));
      xhs[e] = xh;
      rr[e] = __fsub_rn(x[e], xh);
      ferr = __fadd_ru(ferr, resid_err(rr[e], rr[e]));
      if (tensor == 0 || STAGED) packed |= (uint32_t)c << (8 * e);
      else bp[Fp8Layout::VC + vcode_off(r, 4 * lane + e)] = (uint8_t)c;
    }
    if (STAGED && tensor == 1) vst[r * 32 + lane] = packed;
    auto resid_df = [&]() {
#pragma unroll
      for (int e = 0; e < 4; ++e) rdf[e] = residual_df(x[e], -xhs[e], 0.f, 0.f);   // exact: one error-free sum
      return true;
    };
    if (tensor == 0) {
      *reinterpret_cast<uint32_t*>(bp + Fp8Layout::KC + kcode_off(r, 4 * lane)) = packed;
      if (store_witness_fast(bp + Fp8Layout::W, r, rr, ferr, lane, repaired)) continue;
      resid_df();
      if (!store_witness_df(bp + Fp8Layout::W, r, rdf, 0.f, lane, repaired)) {
        double res[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) res[e] = (double)x[e] - (double)xhs[e];
        store_witness(bp + Fp8Layout::W, r, res, lane, repaired);
      }
    } else if (a.vwit && !store_rownorm_fast(vwit_at(a, i, h, t), rr, ferr, lane) && resid_df() &&
               !store_rownorm_df(vwit_at(a, i, h, t), rdf, 0.f, lane)) {
      double res[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) res[e] = (double)x[e] - (double)xhs[e];
      store_rownorm(vwit_at(a, i, h, t), res, lane);
    }
  }
}

// Black-box scheme: the caller's K_hat, V_hat rows rounded to bfloat16 (nearest even) are the
// store; the key witness (and the value witness) are taken against those stored values.
template <typename T>
__device__ __forceinline__ void bbox_token(const WriteArgs& a, uint8_t* bp, int i, int h, int t, size_t row, int lane,
                                           const TokIn<T>& in) {
  const int r = t & 15;
  const bool repaired = exact_side<T>(a, i, h, t, lane, reinterpret_cast<const T*>(a.K) + row);
#pragma unroll
  for (int tensor = 0; tensor < 2; ++tensor) {
    float x[4], y[4];
    (tensor ? in.v : in.k).get(x);
    (tensor ? in.vh : in.kh).get(y);
    const __nv_bfloat162 p01 = __floats2bfloat162_rn(y[0], y[1]), p23 = __floats2bfloat162_rn(y[2], y[3]);
    const float xh[4] = {__low2float(p01), __high2float(p01), __low2float(p23), __high2float(p23)};
    Df rdf[4];
    float rr[4], ferr = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      rr[e] = __fsub_rn(x[e], xh[e]);
      ferr = __fadd_ru(ferr, resid_err(rr[e], rr[e]));
    }
    auto resid_df = [&]() {
#pragma unroll
      for (int e = 0; e < 4; ++e) rdf[e] = residual_df(x[e], -xh[e], 0.f, 0.f);   // exact: one error-free sum
      return true;
    };
    if (tensor == 0) {
      // channels 4 lane .. 4 lane + 3: registers h (e = 0, 1) and h + 2 (e = 2, 3) of one (k-step, lane) slot
      *reinterpret_cast<uint32_t*>(bp + BboxLayout::KH + kbf_off(r, 4 * lane)) = bf2_bits(p01);
      *reinterpret_cast<uint32_t*>(bp + BboxLayout::KH + kbf_off(r, 4 * lane + 2)) = bf2_bits(p23);
      if (store_witness_fast(bp + BboxLayout::W, r, rr, ferr, lane, repaired)) continue;
      resid_df();
      if (!store_witness_df(bp + BboxLayout::W, r, rdf, 0.f, lane, repaired)) {
        double res[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) res[e] = (double)x[e] - (double)xh[e];
        store_witness(bp + BboxLayout::W, r, res, lane, repaired);
      }
    } else {
      __nv_bfloat16* vh = reinterpret_cast<__nv_bfloat16*>(bp + BboxLayout::VH);
      vh[vbf_off(r, 4 * lane) / 2] = __low2bfloat16(p01);
      vh[vbf_off(r, 4 * lane + 1) / 2] = __high2bfloat16(p01);
      vh[vbf_off(r, 4 * lane + 2) / 2] = __low2bfloat16(p23);
      vh[vbf_off(r, 4 * lane + 3) / 2] = __high2bfloat16(p23);
      if (a.vwit && !store_rownorm_fast(vwit_at(a, i, h, t), rr, ferr, lane) && resid_df() &&
          !store_rownorm_df(vwit_at(a, i, h, t), rdf, 0.f, lane)) {
        double res[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) res[e] = (double)x[e] - (double)xh[e];
        store_rownorm(vwit_at(a, i, h, t), res, lane);
      }
    }
  }
}

// Input row (element offset into K, V) of token n of a write that appends n_tok tokens to
// every sequence, sequence-major.
__device__ __forceinline__ size_t uniform_row(const WriteArgs& a, int i, int n, int h) {
  return (((size_t)i * a.n_tok + n) * a.Hkv + h) * kD;
}

// One token of a write into the block image at bp, by scheme (VW: with value witnesses), from
// the lane's inputs `in`; STAGED as for int8_token (the black-box store stages nothing).
template <typename T, int SCH, bool VW, bool STAGED>
__device__ __forceinline__ void write_token(const WriteArgs& a, uint8_t* bp, uint32_t* vst, int i, int h, int t,
                                            size_t row, int lane, const TokIn<T>& in) {
  if constexpr (int8_layout(SCH)) int8_token<T, SCH == kInt8, VW, STAGED>(a, bp, vst, i, h, t, row, lane, in);
  else if constexpr (SCH == kFp8) fp8_token<T, STAGED>(a, bp, vst, i, h, t, row, lane, in);
  else bbox_token<T>(a, bp, i, h, t, row, lane, in);
}
// Load, then write one token straight into its block.
template <typename T, int SCH, bool VW>
__device__ __forceinline__ void write_token_direct(const WriteArgs& a, uint8_t* bp, int i, int h, int t, size_t row,
                                                   int lane) {
  TokIn<T> in;
  in.load(a, row, lane, SCH == kBbox);
  write_token<T, SCH, VW, false>(a, bp, nullptr, i, h, t, row, lane, in);
}


// One warp per (sequence, token, KV head) of tokens tok_begin .. tok_begin + tok_count - 1:
// appends and the parts of a write that do not fill whole blocks.
template <typename T, int SCH, bool VW>
__global__ void __launch_bounds__(128) write_token_kernel(const WriteArgs a) {
  const ChainEntry chain(a.late_wait != 0);
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= a.B * a.tok_count * a.Hkv) return;
  const int h = wid % a.Hkv, n = a.tok_begin + (wid / a.Hkv) % a.tok_count, i = wid / (a.Hkv * a.tok_count);
  const int blk = (a.t0 + n) >> 4;
  constexpr int kBytes = block_bytes(SCH);
  uint8_t* bp = a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, blk) * kBytes;
  write_token_direct<T, SCH, VW>(a, bp, i, h, a.t0 + n, uniform_row(a, i, n, h), lane);
}

// One warp per (sequence, KV head, block) for blocks blk0, blk0 + 1, ... that the write fills
// completely: the warp builds the block's image in shared memory token by token and stores
// it with 16-byte writes.
// The next token's inputs are loaded while a token is quantized.  The INT8 and FP8 value codes
// of the block are staged in natural order (a conflict-free word per lane and token) and then
// packed into their fragment-order words, lane by lane: the word of channel c and lane slot t
// holds tokens 2t, 2t + 1, 2t + 8, 2t + 9.
// Four warps a CTA.  The INT8 and FP8 writers are held to 64 registers a thread, so that the
// shared-memory images, not the registers, bound an SM at seven CTAs (28 warps; 24 at 80
// registers): INT8 bulk writes 0.198 -> 0.214 of HBM at 32k.  Six-warp CTAs (30 warps, the most
// that 48 KB of static shared memory per CTA allows) measured a little slower, and the
// black-box writer is faster at six CTAs of up to 85 registers than at eight of 64.
constexpr int kBlockWriterWarps = 4;
template <typename T, int SCH, bool VW>
__global__ void __launch_bounds__(kBlockWriterWarps * 32, SCH == kBbox ? 6 : 8) write_block_kernel(const WriteArgs a, int blk0, int nblocks) {
  const ChainEntry chain(a.late_wait != 0);
  constexpr int kBytes = block_bytes(SCH);
  constexpr bool kStaged = SCH != kBbox;
  __shared__ __align__(16) uint8_t img[kBlockWriterWarps][kBytes];
  __shared__ uint32_t vstage[kBlockWriterWarps][kStaged ? kBlk * 32 : 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long unit = (long long)blockIdx.x * kBlockWriterWarps + warp;   // (i * Hkv + h) * nblocks + b
  if (unit >= (long long)a.B * a.Hkv * nblocks) return;
  const int b = (int)(unit % nblocks), sh = (int)(unit / nblocks);
  const int i = sh / a.Hkv, h = sh % a.Hkv, blk = blk0 + b;
  uint8_t* im = img[warp];
  uint32_t* vst = vstage[warp];
  TokIn<T> cur, nxt;
  cur.load(a, uniform_row(a, i, blk * kBlk - a.t0, h), lane, SCH == kBbox);
  for (int r = 0; r < kBlk; ++r) {
    const int t = blk * kBlk + r;
    if (r + 1 < kBlk) nxt.load(a, uniform_row(a, i, t + 1 - a.t0, h), lane, SCH == kBbox);
    write_token<T, SCH, VW, kStaged>(a, im, vst, i, h, t, uniform_row(a, i, t - a.t0, h), lane, cur);
    cur = nxt;
  }
  __syncwarp();
  if constexpr (kStaged) {
    constexpr int kVC = SCH == kFp8 ? Fp8Layout::VC : Int8Layout::VC;
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      const uint32_t w0 = vst[(2 * tt) * 32 + lane], w1 = vst[(2 * tt + 1) * 32 + lane];
      const uint32_t w2 = vst[(2 * tt + 8) * 32 + lane], w3 = vst[(2 * tt + 9) * 32 + lane];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t lo = __byte_perm(w0, w1, (uint32_t)(e | ((4 + e) << 4)));
        const uint32_t hi = __byte_perm(w2, w3, (uint32_t)(e | ((4 + e) << 4)));
        *reinterpret_cast<uint32_t*>(im + kVC + vcode_off(2 * tt, 4 * lane + e)) = __byte_perm(lo, hi, 0x5410u);
      }
    }
    __syncwarp();
  }
  uint4* dst = reinterpret_cast<uint4*>(a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, blk) * kBytes);
  const uint4* src = reinterpret_cast<const uint4*>(im);
  for (int k = lane; k < kBytes / 16; k += 32) dst[k] = src[k];
}

// KIVI asymmetric 2-bit of one value against fp16 scale/zero (fp32 steps as the oracle states them).
// ysc = RN(1 / sc): the quotient by div_rn_by, equal to the IEEE one wherever it can move a code.
__device__ __forceinline__ int kivi_code(float x, float zr, float sc, float ysc) {
  if (!(sc > 0.0f)) return 0;
  float v = rintf(div_rn_by(__fsub_rn(x, zr), sc, ysc));
  v = fminf(fmaxf(v, 0.0f), 3.0f);
  return (int)v;
}
__device__ __forceinline__ __half f16_sat_rn(float v) { return __float2half_rn(fminf(fmaxf(v, -65504.0f), 65504.0f)); }

// KIVI values of one token (per 32-channel group) + backing store of its key; bp is the
// token's block in device memory.
template <typename T>
__device__ __forceinline__ void kivi_v_token(const WriteArgs& a, uint8_t* bp, int i, int h, int t, size_t row, int lane) {
  const int r = t & 15;
  exact_side<T>(a, i, h, t, lane, reinterpret_cast<const T*>(a.K) + row);
  float x[4];
  load4f<T>(reinterpret_cast<const T*>(a.V) + row + 4 * lane, x);
  const float mn = grp_min8(fminf(fminf(x[0], x[1]), fminf(x[2], x[3])));
  const float mx = grp_max8(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])));
  const __half sc16 = f16_sat_rn(div_rn_by(__fsub_rn(mx, mn), 3.0f, kInv3));
  const __half zr16 = f16_sat_rn(mn);
  const float sc = __half2float(sc16), zr = __half2float(zr16);
  const float ysc = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
  int codes[4];
  Df rdf[4];
  float err = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int code = kivi_code(x[e], zr, sc, ysc);
    codes[e] = code;
    int off, bit;
    kivi_v_pos(r, 4 * lane + e, off, bit);
    // the word's other fields belong to other tokens and channels: clear this field (a
    // sequence that was reset leaves old bits), then set it
    unsigned int* word = reinterpret_cast<unsigned int*>(bp + KiviLayout::VC + off);
    atomicAnd(word, ~(3u << bit));
    if (code) atomicOr(word, (unsigned int)code << bit);
    // residual x - (zero + scale code): scale code is exact (at most 13 significant bits)
    const float scc = __fmul_rn(sc, (float)code);
    rdf[e] = residual_df(x[e], -zr, -scc, 0.f);
    err = __fadd_ru(err, __fmul_ru(0x1p-46f, __fadd_ru(__fadd_ru(fabsf(x[e]), fabsf(zr)), fabsf(scc))));
  }
  if ((lane & 7) == 0) {
    __half* vp = reinterpret_cast<__half*>(bp + KiviLayout::VP) + (r * 4 + (lane >> 3)) * 2;
    vp[0] = sc16;
    vp[1] = zr16;
  }
  if (a.vwit && !store_rownorm_df(vwit_at(a, i, h, t), rdf, err, lane)) {
    double res[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) res[e] = (double)x[e] - ((double)zr + (double)sc * (double)codes[e]);
    store_rownorm(vwit_at(a, i, h, t), res, lane);
  }
}

template <typename T>
__global__ void __launch_bounds__(128) write_kivi_v_kernel(const WriteArgs a) {
  const ChainEntry chain(a.late_wait != 0);
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= a.B * a.n_tok * a.Hkv) return;
  const int h = wid % a.Hkv, n = (wid / a.Hkv) % a.n_tok, i = wid / (a.Hkv * a.n_tok);
  const int t = a.t0 + n;
  uint8_t* bp = a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, t >> 4) * KiviLayout::BYTES;
  kivi_v_token<T>(a, bp, i, h, t, uniform_row(a, i, n, h), lane);
}

// Ragged appends: sequence seq[k] (k < n_seq) gets its off[k+1] - off[k] tokens, packed from
// input row row0[k] on, at positions t0[k], t0[k] + 1, ...  One warp per (token of the launch,
// KV head); KIVI keys are handled per sequence by write_kivi_k_kernel.
template <typename T, int SCH, bool VW>
__global__ void __launch_bounds__(128) write_ragged_kernel(const WriteArgs a, const RaggedArgs g) {
  pdl_wait();
  pdl_trigger();
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int total = g.off[g.n_seq];
  if (wid >= total * a.Hkv) return;
  const int h = wid % a.Hkv, tok = wid / a.Hkv;
  int lo = 0, hi = g.n_seq - 1;                     // the k with off[k] <= tok < off[k + 1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (g.off[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  const int i = g.seq[lo], t = g.t0[lo] + (tok - g.off[lo]);
  const size_t row = ((size_t)(g.row0[lo] + (tok - g.off[lo])) * a.Hkv + h) * kD;
  uint8_t* bp = a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, t >> 4) * block_bytes(SCH);
  if constexpr (SCH == kKivi) kivi_v_token<T>(a, bp, i, h, t, row, lane);
  else write_token_direct<T, SCH, VW>(a, bp, i, h, t, row, lane);
}

// Per-sequence lengths on the device ([B] of one layer), set from the launch's parameters.
__global__ void __launch_bounds__(128) set_lengths_kernel(const LengthArgs u) {
  pdl_wait();
  pdl_trigger();
  for (int k = threadIdx.x; k < u.n; k += blockDim.x) u.dst[u.idx[k]] = u.len[k];
}

// KIVI keys: one warp per (sequence, KV head, block) this write touches.  Blocks the write
// completes are quantized (block blk0 + blockIdx.y); the block it leaves unfinished is
// launched after them and keeps its new keys exact in the tail, which the first completed
// block may still have to read.
template <typename T>
__global__ void __launch_bounds__(32) write_kivi_k_kernel(const WriteArgs a, int blk0) {
  pdl_wait();
  pdl_trigger();
  const int sh = blockIdx.x, lane = threadIdx.x;       // sh = i * Hkv + h
  const int i = sh / a.Hkv, h = sh % a.Hkv;
  __shared__ unsigned int img[128];                    // K code words of one block
  float* tail = a.kivi_tail + (size_t)sh * kBlk * kD;
  const int t_end = a.t0 + a.n_tok;
  {
    const int blk = blk0 + blockIdx.y;
    const int lo = blk * kBlk;
    if (lo + kBlk > t_end) {   // unfinished block: keep the new keys exact in the tail
      uint8_t* wreg = a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, blk) * KiviLayout::BYTES + KiviLayout::W;
      for (int t = (a.t0 > lo ? a.t0 : lo); t < t_end; ++t) {
        float x[4];
        load4f<T>(reinterpret_cast<const T*>(a.K) + (((size_t)i * a.n_tok + (t - a.t0)) * a.Hkv + h) * kD + 4 * lane, x);
        *reinterpret_cast<float4*>(tail + (t - lo) * kD + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
        // exact keys: zero witness (the row may hold a witness of a sequence that was reset)
        if (lane < kBands) *reinterpret_cast<__half*>(wreg + wit_off(t - lo, lane)) = __float2half_rn(0.f);
      }
      __syncwarp();
      return;
    }
    float x[16][4];
#pragma unroll
    for (int r = 0; r < kBlk; ++r) {
      const int t = lo + r;
      if (t < a.t0) {
        const float4 v = *reinterpret_cast<const float4*>(tail + r * kD + 4 * lane);
        x[r][0] = v.x; x[r][1] = v.y; x[r][2] = v.z; x[r][3] = v.w;
      } else {
        load4f<T>(reinterpret_cast<const T*>(a.K) + (((size_t)i * a.n_tok + (t - a.t0)) * a.Hkv + h) * kD + 4 * lane, x[r]);
      }
    }
    for (int k = lane; k < 128; k += 32) img[k] = 0u;
    __syncwarp();
    uint8_t* bp = a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, blk) * KiviLayout::BYTES;
    __half* ksc = reinterpret_cast<__half*>(bp + KiviLayout::KP);
    __half* kzr = reinterpret_cast<__half*>(bp + KiviLayout::KP + 256);
    float sc[4], zr[4], ysc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float mn = x[0][e], mx = x[0][e];
#pragma unroll
      for (int r = 1; r < kBlk; ++r) { mn = fminf(mn, x[r][e]); mx = fmaxf(mx, x[r][e]); }
      const __half s16 = f16_sat_rn(div_rn_by(__fsub_rn(mx, mn), 3.0f, kInv3));
      const __half z16 = f16_sat_rn(mn);
      const int c = 4 * lane + e;
      ksc[kivi_kparam_idx(c)] = s16;
      kzr[kivi_kparam_idx(c)] = z16;
      sc[e] = __half2float(s16);
      zr[e] = __half2float(z16);
      ysc[e] = sc[e] > 0.0f ? __frcp_rn(sc[e]) : 0.0f;
    }
#pragma unroll
    for (int r = 0; r < kBlk; ++r) {
      int codes[4];
      Df rdf[4];
      float err = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int code = kivi_code(x[r][e], zr[e], sc[e], ysc[e]);
        codes[e] = code;
        // residual x - (zero + scale code): scale code is exact (at most 13 significant bits)
        const float scc = __fmul_rn(sc[e], (float)code);
        rdf[e] = residual_df(x[r][e], -zr[e], -scc, 0.f);
        err = __fadd_ru(err, __fmul_ru(0x1p-46f, __fadd_ru(__fadd_ru(fabsf(x[r][e]), fabsf(zr[e])), fabsf(scc))));
        int off, bit;
        kivi_k_pos(r, 4 * lane + e, off, bit);
        if (code) atomicOr(&img[off / 4], (unsigned int)code << bit);
      }
      if (!store_witness_df(bp + KiviLayout::W, r, rdf, err, lane, false)) {
        double res[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) res[e] = (double)x[r][e] - ((double)zr[e] + (double)sc[e] * (double)codes[e]);
        store_witness(bp + KiviLayout::W, r, res, lane, false);
      }
    }
    __syncwarp();
    for (int k = lane; k < 128; k += 32) reinterpret_cast<unsigned int*>(bp + KiviLayout::KC)[k] = img[k];
    __syncwarp();
  }
}

template <typename K, typename... Extra>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, cudaStream_t st, bool pdl, const WriteArgs& a, Extra... extra) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, a, extra...);
}

// KIVI keys of a write: the blocks it completes, then the unfinished one (if any).
template <typename T>
cudaError_t kivi_keys_t(const WriteArgs& a, cudaStream_t st, bool pdl) {
  cudaError_t e = cudaSuccess;
  const int t_end = a.t0 + a.n_tok, b0 = a.t0 / kBlk, nfull = t_end / kBlk - b0;
  if (nfull > 0) {
    e = launch_pdl(write_kivi_k_kernel<T>, dim3(a.B * a.Hkv, nfull), dim3(32), st, pdl, a, b0);
    if (e != cudaSuccess) return e;
  }
  if (t_end % kBlk) e = launch_pdl(write_kivi_k_kernel<T>, dim3(a.B * a.Hkv, 1), dim3(32), st, pdl, a, t_end / kBlk);
  return e;
}

template <typename T>
cudaError_t launch_t(int scheme, const WriteArgs& a, cudaStream_t st, bool pdl) {
  const int warps = a.B * a.n_tok * a.Hkv;
  const dim3 blocks((warps * 32 + 127) / 128);
  if (scheme != kKivi) {
    // whole blocks through shared-memory images, the rest token by token
    const int t_end = a.t0 + a.n_tok;
    const int lo_full = (a.t0 + kBlk - 1) / kBlk * kBlk, hi_full = t_end / kBlk * kBlk;
    auto tokens = [&](int begin, int count) -> cudaError_t {
      if (count <= 0) return cudaSuccess;
      WriteArgs b = a;
      b.tok_begin = begin;
      b.tok_count = count;
      const dim3 g(((unsigned)(a.B * count * a.Hkv) * 32u + 127u) / 128u);
      const bool vw = a.vwit != nullptr;        // the INT8 writers compile the value witness in or out
      return scheme == kInt8  ? (vw ? launch_pdl(write_token_kernel<T, kInt8, true>, g, dim3(128), st, pdl, b)
                                    : launch_pdl(write_token_kernel<T, kInt8, false>, g, dim3(128), st, pdl, b))
             : scheme == kRtn ? (vw ? launch_pdl(write_token_kernel<T, kRtn, true>, g, dim3(128), st, pdl, b)
                                    : launch_pdl(write_token_kernel<T, kRtn, false>, g, dim3(128), st, pdl, b))
             : scheme == kFp8 ? launch_pdl(write_token_kernel<T, kFp8, false>, g, dim3(128), st, pdl, b)
                              : launch_pdl(write_token_kernel<T, kBbox, false>, g, dim3(128), st, pdl, b);
    };
    if (hi_full <= lo_full) return tokens(0, a.n_tok);
    cudaError_t e = tokens(0, lo_full - a.t0);
    if (e != cudaSuccess) return e;
    const int nblocks = (hi_full - lo_full) / kBlk;
    const dim3 g((unsigned)(((long long)a.B * a.Hkv * nblocks + kBlockWriterWarps - 1) / kBlockWriterWarps));
    const dim3 wb(kBlockWriterWarps * 32);
    const int b0 = lo_full / kBlk;
    const bool vw = a.vwit != nullptr;
    e = scheme == kInt8  ? (vw ? launch_pdl(write_block_kernel<T, kInt8, true>, g, wb, st, pdl, a, b0, nblocks)
                               : launch_pdl(write_block_kernel<T, kInt8, false>, g, wb, st, pdl, a, b0, nblocks))
        : scheme == kRtn ? (vw ? launch_pdl(write_block_kernel<T, kRtn, true>, g, wb, st, pdl, a, b0, nblocks)
                               : launch_pdl(write_block_kernel<T, kRtn, false>, g, wb, st, pdl, a, b0, nblocks))
        : scheme == kFp8 ? launch_pdl(write_block_kernel<T, kFp8, false>, g, wb, st, pdl, a, b0, nblocks)
                         : launch_pdl(write_block_kernel<T, kBbox, false>, g, wb, st, pdl, a, b0, nblocks);
    if (e != cudaSuccess) return e;
    return tokens(hi_full - a.t0, t_end - hi_full);
  }
  cudaError_t e = launch_pdl(write_kivi_v_kernel<T>, blocks, dim3(128), st, pdl, a);
  if (e != cudaSuccess) return e;
  return kivi_keys_t<T>(a, st, pdl);
}

template <typename T>
cudaError_t launch_ragged_t(int scheme, const WriteArgs& a, const RaggedArgs& g, cudaStream_t st, bool pdl) {
  const int total = g.off[g.n_seq];
  if (total == 0) return cudaSuccess;
  const dim3 grid((unsigned)(((long long)total * a.Hkv * 32 + 127) / 128));
  switch (scheme) {
    case kInt8: return a.vwit ? launch_pdl(write_ragged_kernel<T, kInt8, true>, grid, dim3(128), st, pdl, a, g)
                              : launch_pdl(write_ragged_kernel<T, kInt8, false>, grid, dim3(128), st, pdl, a, g);
    case kRtn: return a.vwit ? launch_pdl(write_ragged_kernel<T, kRtn, true>, grid, dim3(128), st, pdl, a, g)
                             : launch_pdl(write_ragged_kernel<T, kRtn, false>, grid, dim3(128), st, pdl, a, g);
    case kFp8: return launch_pdl(write_ragged_kernel<T, kFp8, false>, grid, dim3(128), st, pdl, a, g);
    case kKivi: return launch_pdl(write_ragged_kernel<T, kKivi, false>, grid, dim3(128), st, pdl, a, g);
    default: return launch_pdl(write_ragged_kernel<T, kBbox, false>, grid, dim3(128), st, pdl, a, g);
  }
}

}  // namespace

cudaError_t launch_write_ragged(int scheme, const WriteArgs& a, const RaggedArgs& g, cudaStream_t st, bool pdl) {
  return a.is_bf16 ? launch_ragged_t<__nv_bfloat16>(scheme, a, g, st, pdl) : launch_ragged_t<float>(scheme, a, g, st, pdl);
}

cudaError_t launch_kivi_keys(const WriteArgs& a, cudaStream_t st, bool pdl) {
  if (a.B * a.n_tok * a.Hkv == 0) return cudaSuccess;
  return a.is_bf16 ? kivi_keys_t<__nv_bfloat16>(a, st, pdl) : kivi_keys_t<float>(a, st, pdl);
}

cudaError_t launch_set_lengths(const LengthArgs& u, cudaStream_t st, bool pdl) {
  if (u.n <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, set_lengths_kernel, u);
}

namespace {

// 32-bit mix of a counter (the xorshift-multiply finalizer of MurmurHash3): test inputs only.
__device__ __forceinline__ uint32_t mix32(uint32_t h) {
  h ^= h >> 16; h *= 0x85ebca6bu; h ^= h >> 13; h *= 0xc2b2ae35u; h ^= h >> 16;
  return h;
}

// One CTA per positive fp16 scale (bits 1 .. 0x7BFF): every bf16 x with |x| <= 127.5 s, then
// n_f32 fp32 x = s * u with u drawn in (-127.5, 127.5).  Two more CTAs divide by the constants
// 127 (the INT8 scale) and 3 (the KIVI scale), every finite bf16 x and n_f32 fp32 x drawn over
// fp32's exponent range.  Counts quotients that differ from the IEEE quotient where a code or a
// scale can depend on them (|x / s| >= 2^-25).
__global__ void __launch_bounds__(256) quotient_selftest_kernel(int n_f32, uint32_t seed, unsigned long long* bad) {
  const bool konst = blockIdx.x >= 0x7BFF;
  const float s = konst ? (blockIdx.x == 0x7BFF ? 127.0f : 3.0f) : __half2float(__ushort_as_half((unsigned short)(blockIdx.x + 1)));
  const float y = konst ? (blockIdx.x == 0x7BFF ? kInv127 : kInv3) : __frcp_rn(s);
  const float range = konst ? FLT_MAX : 127.5f * s;
  unsigned long long cnt = 0;
  for (int b = threadIdx.x; b < 65536 + n_f32; b += blockDim.x) {
    float x;
    if (b < 65536) {
      x = __uint_as_float((uint32_t)b << 16);
    } else {
      const uint32_t h = mix32(seed ^ mix32((uint32_t)(blockIdx.x * 0x9E3779B9u) ^ (uint32_t)b));
      if (konst) x = __uint_as_float(h);                         // any bit pattern; inf and NaN skipped
      else x = __fmul_rn(s, __fmul_rn((float)(int)(h >> 8) - 8388608.0f, 0x1.fep-17f));   // u = 127.5 (m - 2^23) / 2^23
    }
    if (!(fabsf(x) <= range)) continue;
    const float want = __fdiv_rn(x, s);
    if (fabsf(want) >= 0x1p-25f && __float_as_uint(div_rn_by(x, s, y)) != __float_as_uint(want)) ++cnt;
  }
  if (cnt) atomicAdd(bad, cnt);
}

}  // namespace

cudaError_t run_quotient_selftest(int n_f32, uint64_t seed, unsigned long long* mismatches, cudaStream_t st) {
  unsigned long long* d = nullptr;
  cudaError_t e = cudaMalloc(&d, sizeof(unsigned long long));
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(d, 0, sizeof(unsigned long long), st);
  if (e == cudaSuccess) {
    quotient_selftest_kernel<<<0x7BFF + 2, 256, 0, st>>>(n_f32, (uint32_t)(seed ^ (seed >> 32)), d);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpyAsync(mismatches, d, sizeof(unsigned long long), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(d);
  return e;
}

void philox_round_keys(uint64_t seed, uint32_t (&rk0)[10], uint32_t (&rk1)[10]) {
  uint32_t k0 = (uint32_t)(seed & 0xFFFFFFFFull), k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    rk0[r] = k0;
    rk1[r] = k1;
  }
}

cudaError_t launch_write(int scheme, const WriteArgs& a, cudaStream_t st, bool pdl) {
  if (a.B * a.n_tok * a.Hkv == 0) return cudaSuccess;
  return a.is_bf16 ? launch_t<__nv_bfloat16>(scheme, a, st, pdl) : launch_t<float>(scheme, a, st, pdl);
}

}  // namespace witcert
