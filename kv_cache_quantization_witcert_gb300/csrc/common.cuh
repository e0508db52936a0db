// Device-side building blocks shared by the write, decode, gate and export kernels.
//
// Cache layout in HBM.  For every (layer, sequence, KV head) the cache is one
// contiguous stream of 16-token blocks; a block holds everything a decode
// needs for those 16 tokens, so one bulk copy stages it:
//
//   INT8_DITHER (4864 B = 16 x 304):  K codes 2048 | V codes 2048 | K scales 128 | V scales 128 | witness 512
//   FP8_E4M3    (4608 B = 16 x 288):  K codes 2048 | V codes 2048 | witness 512
//   KIVI2       (2304 B = 16 x 144):  K codes 512 | K scale,zero 512 | V codes 512 | V scale,zero 256 | witness 512
//   BLACKBOX    (8704 B = 16 x 544):  K_hat bf16 4096 | V_hat bf16 4096 | witness 512
//
// With the value witness on, a separate array holds one fp16 norm per token:
// 32 bytes per block, [B][Hkv][nblk_max][16] per layer.  A paged cache keeps the blocks
// in a pool of pages instead (see block_index); every other array stays per sequence.
//
// Codes are stored in "fragment order": the byte a lane of a warp needs for
// the A operand of mma.m16n8k16 sits where one 16-byte shared-memory load per
// lane fetches it without bank conflicts.  The index functions below are the
// single definition of that order; export kernels invert them.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace witcert {

constexpr int kD = 128;
constexpr int kBlk = 16;
constexpr int kBands = 16;
constexpr int kGroupCh = 32;
constexpr int kGroups = 4;
constexpr int kMaxGroupHeads = 8;

enum SchemeId : int { kInt8 = 0, kFp8 = 1, kKivi = 2, kRtn = 3, kBbox = 4 };
// INT8 round-to-nearest (kRtn) keeps the dithered scheme's block layout without the dither.
__host__ __device__ constexpr bool int8_layout(int scheme) { return scheme == kInt8 || scheme == kRtn; }

struct Int8Layout { static constexpr int KC = 0, VC = 2048, KS = 4096, VS = 4224, W = 4352, BYTES = 4864; };
struct Fp8Layout  { static constexpr int KC = 0, VC = 2048, W = 4096, BYTES = 4608; };
struct KiviLayout { static constexpr int KC = 0, KP = 512, VC = 1024, VP = 1536, W = 1792, BYTES = 2304; };
struct BboxLayout { static constexpr int KH = 0, VH = 4096, W = 8192, BYTES = 8704; };
constexpr int kVwBytes = kBlk * 2;   // value witnesses of one block

__host__ __device__ constexpr int block_bytes(int scheme) {
  return int8_layout(scheme) ? Int8Layout::BYTES
         : scheme == kFp8    ? Fp8Layout::BYTES
         : scheme == kKivi   ? KiviLayout::BYTES
                             : BboxLayout::BYTES;
}
__host__ __device__ constexpr int witness_off(int scheme) {
  return int8_layout(scheme) ? Int8Layout::W : scheme == kFp8 ? Fp8Layout::W : scheme == kKivi ? KiviLayout::W : BboxLayout::W;
}

// Index of block b of (sequence i, KV head h) in a layer's block store: [B][Hkv][nblk_max]
// blocks in a contiguous store, or page table[i][b] of a paged store ([pages][Hkv] blocks;
// a page holds one 16-token block of every KV head of one sequence).
__host__ __device__ inline size_t block_index(const int32_t* table, int Hkv, int nblk_max, int i, int h, int b) {
  return table ? (size_t)table[(size_t)i * nblk_max + b] * Hkv + h : ((size_t)i * Hkv + h) * nblk_max + b;
}

// ------------------------------------------------------------------ fragment-order index maps
// Lane L = 4g + t (g = L>>2, t = L&3).  mma.m16n8k16 A fragment of lane L:
//   R0 = row g,   k {2t, 2t+1}     R1 = row g+8, k {2t, 2t+1}
//   R2 = row g,   k {2t+8, 2t+9}   R3 = row g+8, k {2t+8, 2t+9}
// and B fragment: R0 = k {2t, 2t+1}, col g;  R1 = k {2t+8, 2t+9}, col g.
// The k index of a 16-wide step is mapped to four consecutive physical
// elements per lane: k 2t,2t+1 -> 4t,4t+1 and k 2t+8,2t+9 -> 4t+2,4t+3.

// 1-byte K code of token r (0..15), channel c: QK^T with tokens as rows.
__host__ __device__ inline int kcode_off(int r, int c) {
  int g = r & 7, h = r >> 3, kk = c >> 4, t = (c >> 2) & 3, e = c & 3;
  int L = 4 * g + t, j = kk >> 1, slot = ((kk & 1) << 1) | h;
  return j * 512 + L * 16 + slot * 4 + e;
}
// Token r of a block as a k index of the P.V product (tokens as k, natural order):
// lane t holds k 2t, 2t+1 in its first register and 2t+8, 2t+9 in its second, the
// layout a transposed (movmatrix) softmax fragment arrives in.  Slot e = 0..3 of
// lane t is token 2t, 2t+1, 2t+8, 2t+9.
__host__ __device__ inline int pv_lane(int r) { return (r & 7) >> 1; }
__host__ __device__ inline int pv_slot(int r) { return (r & 1) | ((r >> 3) << 1); }
// 1-byte V code: PV^T with channels as rows and tokens as k.
__host__ __device__ inline int vcode_off(int r, int c) {
  int mt = c >> 4, g = c & 7, h = (c >> 3) & 1, t = pv_lane(r), e = pv_slot(r);
  int L = 4 * g + t, j = mt >> 1, slot = ((mt & 1) << 1) | h;
  return j * 512 + L * 16 + slot * 4 + e;
}
// fp16 witness of token r, band b: A operand of the Tier A product (bands as k).
// Lane t's k indices 2t, 2t+1, 2t+8, 2t+9 carry bands t, t+4, t+8, t+12: the bands
// whose dims (4b..4b+3 and 64+4b..64+4b+3) sit in that lane's query fragment.
__host__ __device__ inline int wit_off(int r, int b) {
  int g = r & 7, h = r >> 3, t = b & 3, m = b >> 2, hi = m >> 1, e = m & 1;
  int L = 4 * g + t, reg = h + 2 * hi;
  return L * 16 + reg * 4 + e * 2;
}
// fp16 INT8 value scale of token r, group G: stored group-major, tokens in P.V slot
// order, so the four scales a lane needs for the P.V operand are adjacent.
__host__ __device__ inline int vscale_off(int r, int G) { return (G * 16 + 4 * pv_lane(r) + pv_slot(r)) * 2; }
// 2-bit KIVI codes: word (byte offset) and bit position.  Each 32-bit word holds
// eight fp16x2 register pairs; pair p keeps its two codes at bits 2p and 16+2p.
__host__ __device__ inline void kivi_k_pos(int r, int c, int& word_off, int& bit) {
  int g = r & 7, h = r >> 3, kk = c >> 4, t = (c >> 2) & 3, e = c & 3;
  int L = 4 * g + t, j = kk >> 1, reg = h + 2 * (e >> 1), p = (kk & 1) * 4 + reg;
  word_off = L * 16 + j * 4;
  bit = 2 * p + 16 * (e & 1);
}
__host__ __device__ inline void kivi_v_pos(int r, int c, int& word_off, int& bit) {
  int mt = c >> 4, g = c & 7, h = (c >> 3) & 1, t = pv_lane(r), e = pv_slot(r);
  int L = 4 * g + t, j = mt >> 1, reg = h + 2 * (e >> 1), p = (mt & 1) * 4 + reg;
  word_off = L * 16 + j * 4;
  bit = 2 * p + 16 * (e & 1);
}
// bf16 key of token r, channel c (black-box store): the QK A operand with two-byte
// elements, 16 bytes per (k-step, lane): register h + 2 (e >> 1), half e & 1.
__host__ __device__ inline int kbf_off(int r, int c) {
  int g = r & 7, h = r >> 3, kk = c >> 4, t = (c >> 2) & 3, e = c & 3;
  return (kk * 32 + 4 * g + t) * 16 + (h + 2 * (e >> 1)) * 4 + (e & 1) * 2;
}
// bf16 value of token r, channel c: the P.V A operand (channels as rows, tokens as k),
// 16 bytes per (m-tile, lane).
__host__ __device__ inline int vbf_off(int r, int c) {
  int mt = c >> 4, g = c & 7, h = (c >> 3) & 1, t = pv_lane(r), e = pv_slot(r);
  return (mt * 32 + 4 * g + t) * 16 + (h + 2 * (e >> 1)) * 4 + (e & 1) * 2;
}
// KIVI K per-channel scale (fp16) index; the zero point sits 256 bytes later.
__host__ __device__ inline int kivi_kparam_idx(int c) { return ((c >> 2) & 3) * 32 + (c >> 4) * 4 + (c & 3); }

// ------------------------------------------------------------------ Philox4x32-10 dither
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}
// xi = (u >> 8) * 2^-24 - 1/2, exact in fp32.
__device__ __forceinline__ float xi_from_word(uint32_t u) {
  return __fadd_rn(__fmul_rn(__uint2float_rn(u >> 8), 5.9604644775390625e-8f), -0.5f);
}
// Dither of channels 4*quad .. 4*quad+3 of token position t.
__device__ __forceinline__ float4 dither4(uint64_t seed, int layer, int kvh, int t, int quad, int tensor) {
  uint4 u = philox4x32_10(make_uint4((uint32_t)t, (uint32_t)quad | ((uint32_t)tensor << 16),
                                     (uint32_t)kvh | ((uint32_t)layer << 16), 0u),
                          (uint32_t)(seed & 0xFFFFFFFFull), (uint32_t)(seed >> 32));
  return make_float4(xi_from_word(u.x), xi_from_word(u.y), xi_from_word(u.z), xi_from_word(u.w));
}

// Philox with the ten round keys precomputed (k0 + r*0x9E3779B9, k1 + r*0xBB67AE85):
// the keys sit in kernel parameters and enter the XORs as constant operands.
__device__ __forceinline__ uint4 philox4x32_10_rk(uint4 c, const uint32_t (&rk0)[10], const uint32_t (&rk1)[10]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ rk0[r], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ rk1[r], (uint32_t)p0);
  }
  return c;
}
__device__ __forceinline__ float4 dither4_rk(const uint32_t (&rk0)[10], const uint32_t (&rk1)[10], int layer, int kvh,
                                             int t, int quad, int tensor) {
  const uint4 u = philox4x32_10_rk(make_uint4((uint32_t)t, (uint32_t)quad | ((uint32_t)tensor << 16),
                                              (uint32_t)kvh | ((uint32_t)layer << 16), 0u), rk0, rk1);
  return make_float4(xi_from_word(u.x), xi_from_word(u.y), xi_from_word(u.z), xi_from_word(u.w));
}

// Negated dither -xi = 1/2 - (u >> 8) * 2^-24 in one FFMA (exact: 24-bit integer, power-of-two scale).
__device__ __forceinline__ float neg_xi_from_word(uint32_t u) {
  return __fmaf_rn(__uint2float_rn(u >> 8), -5.9604644775390625e-8f, 0.5f);
}
__device__ __forceinline__ float4 neg_dither4_rk(const uint32_t (&rk0)[10], const uint32_t (&rk1)[10], int layer,
                                                 int kvh, int t, int quad, int tensor) {
  const uint4 u = philox4x32_10_rk(make_uint4((uint32_t)t, (uint32_t)quad | ((uint32_t)tensor << 16),
                                              (uint32_t)kvh | ((uint32_t)layer << 16), 0u), rk0, rk1);
  return make_float4(neg_xi_from_word(u.x), neg_xi_from_word(u.y), neg_xi_from_word(u.z), neg_xi_from_word(u.w));
}

// 2^x on the special-function unit (relative error about 2^-22; -inf -> +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch: wait for the preceding kernel on the stream (its
// memory is then visible), then let the next kernel start its own prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ------------------------------------------------------------------ tensor-core product
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Transpose of an 8x8 fp16 matrix held as mma fragments (lane 4g + t holds row g,
// columns 2t, 2t+1; afterwards it holds row g of the transpose).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// ------------------------------------------------------------------ small conversions
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) { return h2_bits(__halves2half2(lo, hi)); }
__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Two biased INT8 codes (code + 128 in bytes b, b+1 of w) -> exact fp16x2 codes.
// 0x64XX is the fp16 1024 + XX; subtracting 1152 = 1024 + 128 leaves the code.
__device__ __forceinline__ uint32_t i8x2_lo(uint32_t w) {
  return h2_bits(__hsub2(bits_h2(__byte_perm(w, 0x64646464u, 0x4140u)), __half2half2(__ushort_as_half(0x6480))));
}
__device__ __forceinline__ uint32_t i8x2_hi(uint32_t w) {
  return h2_bits(__hsub2(bits_h2(__byte_perm(w, 0x64646464u, 0x4342u)), __half2half2(__ushort_as_half(0x6480))));
}
// Two E4M3 codes -> fp16x2 (every E4M3 value is exact in fp16).
__device__ __forceinline__ uint32_t e4m3x2_lo(uint32_t w) {
  __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
  return (uint32_t)r.x | ((uint32_t)r.y << 16);
}
__device__ __forceinline__ uint32_t e4m3x2_hi(uint32_t w) {
  __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  return (uint32_t)r.x | ((uint32_t)r.y << 16);
}
// Two 2-bit codes at bits 2p and 16+2p of w -> exact fp16x2.
__device__ __forceinline__ uint32_t u2x2(uint32_t w, int p) {
  uint32_t x = ((w >> (2 * p)) & 0x00030003u) | 0x64006400u;
  return h2_bits(__hsub2(bits_h2(x), __half2half2(__ushort_as_half(0x6400))));
}

// Split an fp32 value into fp16 hi + lo with hi + lo == v to ~22 bits.
__device__ __forceinline__ void split_h(float v, __half& hi, __half& lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// expm1 for c >= 0 with small relative error: Taylor-Horner below 1/2, exp - 1 above.
__device__ __forceinline__ float expm1_pos(float c) {
  if (c < 0.5f) {
    float s = 1.0f + c * (1.0f / 8.0f);
    s = 1.0f + c * (1.0f / 7.0f) * s;
    s = 1.0f + c * (1.0f / 6.0f) * s;
    s = 1.0f + c * (1.0f / 5.0f) * s;
    s = 1.0f + c * (1.0f / 4.0f) * s;
    s = 1.0f + c * (1.0f / 3.0f) * s;
    s = 1.0f + c * 0.5f * s;
    return c * s;
  }
  return exp2f(c * 1.4426950408889634f) - 1.0f;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded mbarrier wait: returns false once `limit_ns` of wall time has passed.  The
// clock is read only when the first attempt does not find the phase complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
// One-dimensional bulk copy global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Hint: bring `bytes` (a multiple of 16) at a 16-byte aligned global address into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

}  // namespace witcert
