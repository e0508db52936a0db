// Merge of split-KV partial states and the decode launchers (split kernel in decode_split.cuh).
#include <atomic>
#include <cmath>
#include <mutex>

#include "decode_split.cuh"

namespace witcert {

namespace {

// One CTA of kMergeWarps warps per (sequence, query head).  Warp w folds splits w,
// w + kMergeWarps, ... into a running (max, Z, S_A, S_B, S_V, values) with online rescaling, so
// that all its record loads are independent of one another; the warps' states meet in shared
// memory, where thread j finishes channel j.  Then the meters and the block risks.
//
// The records' maxima are integers (log2 units), so every rescale is an exact power of two; the
// sums are Kahan pairs within a warp and meet across warps through two-sums, and they leave their
// pairs rounded down (Z) or up (S_X) before the quotient D = S_X / Z, its margin and D + D^2/2,
// all rounded up.
constexpr int kMergeWarps = 8;

__device__ __forceinline__ void kahan_add(float& hi, float& lo, float x) {
  const float y = x + lo;
  const float t = hi + y;
  lo = y - (t - hi);
  hi = t;
}

// D = S / Z with the meters' margin, rounded up; D + D^2 / 2 rounded up.
__device__ __forceinline__ float meter_ratio(float S_hi, float S_lo, float Z_dn) {
  const float S_up = __fadd_ru(S_hi, S_lo);
  if (!(S_up > 0.f) || !(Z_dn > 0.f)) return 0.f;
  return __fadd_ru(__fmul_ru(__fdiv_ru(S_up, Z_dn), kMeterMargin), kMeterFloor);
}
__device__ __forceinline__ float meter_raw(float D) { return __fmaf_ru(__fmul_ru(0.5f, D), D, D); }

template <bool INT8, bool RISK>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const DecodeArgs p) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_hdr[kMergeWarps][9];       // M, then (hi, lo) of Z, S_A, S_B, S_V
  __shared__ __align__(16) float s_acc[kMergeWarps][kD];
  const int cell = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* recs = p.part + (size_t)cell * p.n_splits * kPartStride;
  const int ns = p.n_splits;
  float M = -INFINITY, Zh = 0.f, Zl = 0.f, Ah = 0.f, Al = 0.f, Bh = 0.f, Bl = 0.f, Vh = 0.f, Vl = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int s = warp; s < ns; s += kMergeWarps) {
    const float* r = recs + (size_t)s * kPartStride;
    const float4 h = *reinterpret_cast<const float4*>(r);           // m, Z, S_A, S_B of the split
    const float sv = r[4];                                          // S_V
    const float4 a = *reinterpret_cast<const float4*>(r + kPartAcc + 4 * lane);
    if (h.x > M) {                                                  // same for every lane
      const float k = M - h.x;                                      // -inf while M is
      const float sd = pow2_dn(k), su = pow2_up(k);
      Zh = __fmul_rd(Zh, sd); Zl = __fmul_rd(Zl, sd);
      Ah = __fmul_ru(Ah, su); Al = __fmul_ru(Al, su);
      Bh = __fmul_ru(Bh, su); Bl = __fmul_ru(Bl, su);
      Vh = __fmul_ru(Vh, su); Vl = __fmul_ru(Vl, su);
      acc.x *= sd; acc.y *= sd; acc.z *= sd; acc.w *= sd;
      M = h.x;
    }
    const float k = h.x == M ? 0.f : h.x - M;                       // -inf for an empty split
    const float fd = pow2_dn(k), fu = pow2_up(k);
    kahan_add(Zh, Zl, __fmul_rd(fd, h.y));
    kahan_add(Ah, Al, __fmul_ru(fu, h.z));
    kahan_add(Bh, Bl, __fmul_ru(fu, h.w));
    kahan_add(Vh, Vl, __fmul_ru(fu, sv));
    acc.x = fmaf(fd, a.x, acc.x); acc.y = fmaf(fd, a.y, acc.y); acc.z = fmaf(fd, a.z, acc.z); acc.w = fmaf(fd, a.w, acc.w);
  }
  if (lane == 0) {
    float* hw = s_hdr[warp];
    hw[0] = M; hw[1] = Zh; hw[2] = Zl; hw[3] = Ah; hw[4] = Al; hw[5] = Bh; hw[6] = Bl; hw[7] = Vh; hw[8] = Vl;
  }
  *reinterpret_cast<float4*>(&s_acc[warp][4 * lane]) = acc;
  __syncthreads();
  // the warps' states meet at the largest maximum.  Every thread forms Z (the same arithmetic in
  // every thread, so the same value) and its output channel; warp 0 forms the S sums and the
  // meters without holding up the output.
  float Mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) Mx = fmaxf(Mx, s_hdr[w][0]);
  float fw[kMergeWarps];
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) fw[w] = Mx == -INFINITY ? 0.f : pow2_dn(s_hdr[w][0] == Mx ? 0.f : s_hdr[w][0] - Mx);
  float Zsh = 0.f, Zsl = 0.f, o = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) {
    pair_add(Zsh, Zsl, __fmul_rd(fw[w], s_hdr[w][1]), __fmul_rd(fw[w], s_hdr[w][2]));
    if (threadIdx.x < kD) o = fmaf(fw[w], s_acc[w][threadIdx.x], o);
  }
  const float Zt = Zsh + Zsl, Zdn = __fadd_rd(Zsh, Zsl);
  // warp 0: lane 8q + w (q = 1, 2, 3: S_A, S_B, S_V) holds warp w's pair of that sum, scaled exactly
  // to Mx (rounded up where the scale leaves fp32's normal range); three rounds of two-sums add
  // the warps, then the first lane of each sum forms its meter against Z
  if (warp == 0) {
    const int q = lane >> 3, w = lane & 7;
    const float* hw = s_hdr[w];
    const float fu = Mx == -INFINITY ? 0.f : pow2_up(hw[0] == Mx ? 0.f : hw[0] - Mx);
    float hi = 0.f, lo = 0.f;
    if (q > 0) { hi = __fmul_ru(fu, hw[2 * q + 1]); lo = __fmul_ru(fu, hw[2 * q + 2]); }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
      const float ohi = __shfl_xor_sync(0xffffffffu, hi, m), olo = __shfl_xor_sync(0xffffffffu, lo, m);
      pair_add(hi, lo, ohi, olo);
    }
    if (p.part_out) {         // context-parallel shard: the cell's combined record, unnormalized
      float* rec = p.part_out + (size_t)cell * kPartStride;
      if (lane == 0) { rec[0] = Mx; rec[1] = Zdn; rec[5] = 0.f; rec[6] = 0.f; rec[7] = 0.f; }
      if (w == 0 && q > 0) rec[1 + q] = __fadd_ru(hi, lo);
    } else if (p.meter && w == 0 && q > 0) {
      const float D = meter_ratio(hi, lo, Zdn);
      if (q == 3) {
        if (p.meter_v) p.meter_v[cell] = D;                       // E_V = S_V / Z, rounded up
      } else if (q == 1) {
        const float rawA = meter_raw(D);
        if (p.raw_a) p.raw_a[cell] = rawA;
        if (p.meter_a) p.meter_a[cell] = fminf(1.0f, rawA);
      } else {
        const float rawB = INT8 ? meter_raw(D) : NAN;
        if (p.raw_b) p.raw_b[cell] = rawB;
        if (p.meter_b) p.meter_b[cell] = INT8 ? fminf(1.0f, rawB) : NAN;
      }
    }
  }
  if (p.part_out) {
    if (threadIdx.x < kD) p.part_out[(size_t)cell * kPartStride + kPartAcc + threadIdx.x] = o;
    return;
  }
  const float inv = Zt > 0.f ? 1.0f / Zt : 0.f;
  if (threadIdx.x < kD) p.out[(size_t)cell * kD + threadIdx.x] = o * inv;
  if (!p.meter) return;
  if (RISK) {
    // block share of D: r 2^(m_blk - M) / Z with the meters' margin, rounded up
    const int nblk = (p.S + kBlk - 1) / kBlk;
    const int S_c = p.seq_len ? p.seq_len[cell / p.Hq] : p.S;      // this cell's sequence
    const int nblk_c = (S_c + kBlk - 1) / kBlk;
    const float2* rr = p.risk_raw + (size_t)cell * p.nblk_max;
    float* ro = p.risk + (size_t)cell * p.nblk_max;
    // margin / Z rounded up once: products of upward-rounded positive factors stay above
    const float scale = Zdn > 0.f ? __fdiv_ru(kMeterMargin, Zdn) : 0.f;
    for (int b = threadIdx.x; b < nblk; b += kMergeWarps * 32) {
      const float2 v = b < nblk_c ? rr[b] : make_float2(0.f, 0.f);
      float r = 0.f;
      if (v.y > 0.f && Zdn > 0.f) {
        const float k = v.x == Mx ? 0.f : v.x - Mx;
        r = __fadd_ru(__fmul_ru(__fmul_ru(v.y, pow2_up(k)), scale), kMeterFloor);
      }
      ro[b] = r;
    }
  }
}

// Sequences (warps) per split CTA.  The dithered scheme rounds the batch up to the next width, so
// that all of it shares one CTA's dither (the dither of a block costs its CTA about 2000 warp
// instructions, however many of its warps use it): at 32k, B = 3 / 6 / 12 run at 0.31 / 0.42 /
// 0.62 of HBM this way against 0.18 / 0.31 / 0.43 in CTAs of 2 / 4 / 8 sequences.
int seqs_per_cta_for(int scheme, int B) {
  const int cap = scheme == kBbox ? 8 : 16;
  int n = B >= 16 ? 16 : B >= 8 ? 8 : B >= 4 ? 4 : B >= 2 ? 2 : 1;
  if (scheme == kInt8 && n < B) n *= 2;
  return n < cap ? n : cap;
}

cudaError_t dispatch_scheme(int scheme, const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ) {
  switch (scheme) {
    case kInt8: return decode_split_int8(a, grid, st, pdl, occ);
    case kRtn: return decode_split_rtn(a, grid, st, pdl, occ);
    case kFp8: return decode_split_fp8(a, grid, st, pdl, occ);
    case kKivi: return decode_split_kivi(a, grid, st, pdl, occ);
    default: return decode_split_bbox(a, grid, st, pdl, occ);
  }
}

}  // namespace

// ------------------------------------------------------------------ scratch without allocation
// Split partials of witcert_decode_noalloc live in this array, which every GPU that
// loads the library holds until the process exits.  Host code must not pass the
// symbol itself to a kernel (on the host it names a stand-in, not device memory):
// its device address is looked up once per device below.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) float g_split_scratch[kStaticScratchBytes / sizeof(float)];

cudaError_t decode_static_scratch(float** ptr, size_t* bytes) {
  static std::mutex mu;
  static float* addr[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float*>(p);
  }
  *ptr = addr[dev];
  *bytes = kStaticScratchBytes;
  return cudaSuccess;
}

cudaError_t launch_merge_records(int scheme, const DecodeArgs& a, cudaStream_t st) {
  const dim3 mg(a.B * a.Hq);
  return scheme == kInt8 ? launch_pdl(decode_merge_kernel<true, false>, mg, dim3(kMergeWarps * 32), 0, st, false, a)
                         : launch_pdl(decode_merge_kernel<false, false>, mg, dim3(kMergeWarps * 32), 0, st, false, a);
}

int decode_ctas_per_sm(int scheme, const DecodeArgs& a0) {
  DecodeArgs a = a0;
  a.seqs_per_cta = seqs_per_cta_for(scheme, a.B);
  int n = 0;
  const cudaError_t e = dispatch_scheme(scheme, a, dim3(1), nullptr, false, &n);
  return e == cudaSuccess && n > 0 ? n : 1;
}

// Splits per (KV head, sequence group): the fewest that fill the GPU's CTA slots
// (per_sm resident CTAs on each of sm_count SMs) to at least 90% in whole waves, so that
// no wave runs with most SMs idle.
int decode_auto_splits(int scheme, int B, int Hkv, int nblk, int sm_count, int per_sm) {
  const int spc = seqs_per_cta_for(scheme, B);
  const long long units = (long long)Hkv * ((B + spc - 1) / spc);
  const long long slots = (long long)sm_count * (per_sm > 0 ? per_sm : 1);
  long long best = 1;
  double best_eff = -1.0;
  for (int w = 1; w <= 4; ++w) {
    long long s = w * slots / units;
    if (s < 1) s = 1;
    if (s > nblk) s = nblk;
    const long long ctas = units * s, waves = (ctas + slots - 1) / slots;
    const double eff = (double)ctas / (double)(waves * slots);
    if (eff > best_eff + 1e-9) { best_eff = eff; best = s; }
    if (eff >= 0.9 || s == nblk) break;
  }
  return (int)best;
}

cudaError_t launch_decode(int scheme, const DecodeArgs& a0, int sm_count, cudaStream_t st,
                          cudaEvent_t split_start, cudaEvent_t split_stop, bool pdl_allowed) {
  (void)sm_count;
  DecodeArgs a = a0;
  a.seqs_per_cta = seqs_per_cta_for(scheme, a.B);
  const int groups = (a.B + a.seqs_per_cta - 1) / a.seqs_per_cta;
  dim3 grid(a.n_splits, a.Hkv, groups);
  // event boundaries around a timed split (and an event wait before it) get a plain launch
  const bool pdl = pdl_allowed && split_start == nullptr;
  cudaError_t e = split_start ? cudaEventRecord(split_start, st) : cudaSuccess;
  if (e != cudaSuccess) return e;
  e = dispatch_scheme(scheme, a, grid, st, pdl, nullptr);
  if (e != cudaSuccess) return e;
  if (split_stop && (e = cudaEventRecord(split_stop, st)) != cudaSuccess) return e;
  const dim3 mg(a.B * a.Hq);
  const bool risk = a.risk_raw != nullptr && a.meter;
  if (scheme == kInt8)
    e = risk ? launch_pdl(decode_merge_kernel<true, true>, mg, dim3(kMergeWarps * 32), 0, st, pdl_allowed, a)
             : launch_pdl(decode_merge_kernel<true, false>, mg, dim3(kMergeWarps * 32), 0, st, pdl_allowed, a);
  else
    e = risk ? launch_pdl(decode_merge_kernel<false, true>, mg, dim3(kMergeWarps * 32), 0, st, pdl_allowed, a)
             : launch_pdl(decode_merge_kernel<false, false>, mg, dim3(kMergeWarps * 32), 0, st, pdl_allowed, a);
  return e;
}

}  // namespace witcert
