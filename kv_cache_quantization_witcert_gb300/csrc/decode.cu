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
constexpr int kMergeWarps = 8;

template <bool INT8, bool RISK>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const DecodeArgs p) {
  pdl_wait();
  pdl_trigger();
  __shared__ float4 s_hdr[kMergeWarps];
  __shared__ float s_sv[kMergeWarps];
  __shared__ __align__(16) float s_acc[kMergeWarps][kD];
  const int cell = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* recs = p.part + (size_t)cell * p.n_splits * kPartStride;
  const int ns = p.n_splits;
  float M = -INFINITY, Z = 0.f, SA = 0.f, SB = 0.f, SV = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int s = warp; s < ns; s += kMergeWarps) {
    const float* r = recs + (size_t)s * kPartStride;
    const float4 h = *reinterpret_cast<const float4*>(r);           // m, Z, S_A, S_B of the split
    const float sv = r[4];                                          // S_V
    const float4 a = *reinterpret_cast<const float4*>(r + kPartAcc + 4 * lane);
    if (h.x > M) {                                                  // same for every lane
      const float sc = M == -INFINITY ? 0.f : ex2(M - h.x);
      Z *= sc; SA *= sc; SB *= sc; SV *= sc;
      acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
      M = h.x;
    }
    const float f = h.x == -INFINITY ? 0.f : ex2(h.x - M);
    Z = fmaf(f, h.y, Z); SA = fmaf(f, h.z, SA); SB = fmaf(f, h.w, SB); SV = fmaf(f, sv, SV);
    acc.x = fmaf(f, a.x, acc.x); acc.y = fmaf(f, a.y, acc.y); acc.z = fmaf(f, a.z, acc.z); acc.w = fmaf(f, a.w, acc.w);
  }
  if (lane == 0) { s_hdr[warp] = make_float4(M, Z, SA, SB); s_sv[warp] = SV; }
  *reinterpret_cast<float4*>(&s_acc[warp][4 * lane]) = acc;
  __syncthreads();
  float Mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) Mx = fmaxf(Mx, s_hdr[w].x);
  float Zt = 0.f, SAt = 0.f, SBt = 0.f, SVt = 0.f, o = 0.f;
  if (Mx != -INFINITY) {
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      const float4 hw = s_hdr[w];
      const float wt = hw.x == -INFINITY ? 0.f : ex2(hw.x - Mx);
      Zt = fmaf(wt, hw.y, Zt); SAt = fmaf(wt, hw.z, SAt); SBt = fmaf(wt, hw.w, SBt); SVt = fmaf(wt, s_sv[w], SVt);
      if (threadIdx.x < kD) o = fmaf(wt, s_acc[w][threadIdx.x], o);
    }
  }
  if (p.part_out) {           // context-parallel shard: the cell's combined record, unnormalized
    float* rec = p.part_out + (size_t)cell * kPartStride;
    if (threadIdx.x == 0) {
      *reinterpret_cast<float4*>(rec) = make_float4(Mx, Zt, SAt, SBt);
      *reinterpret_cast<float4*>(rec + 4) = make_float4(SVt, 0.f, 0.f, 0.f);
    }
    if (threadIdx.x < kD) rec[kPartAcc + threadIdx.x] = o;
    return;
  }
  const float inv = Zt > 0.f ? 1.0f / Zt : 0.f;
  if (threadIdx.x < kD) p.out[(size_t)cell * kD + threadIdx.x] = o * inv;
  if (!p.meter) return;
  if (threadIdx.x == 0 && p.meter_v)    // E_V = S_V / Z, rounded up with the meters' margin
    p.meter_v[cell] = Zt > 0.f ? __fmul_ru(__fdiv_ru(SVt, Zt), kMeterMargin) : 0.f;
  if (threadIdx.x == 0) {
    const float DA = Zt > 0.f ? __fmul_ru(__fdiv_ru(SAt, Zt), kMeterMargin) : 0.f;
    const float rawA = __fmaf_ru(__fmul_ru(0.5f, DA), DA, DA);
    if (p.raw_a) p.raw_a[cell] = rawA;
    if (p.meter_a) p.meter_a[cell] = fminf(1.0f, rawA);
    float rawB = NAN;
    if (INT8) {
      const float DB = Zt > 0.f ? __fmul_ru(__fdiv_ru(SBt, Zt), kMeterMargin) : 0.f;
      rawB = __fmaf_ru(__fmul_ru(0.5f, DB), DB, DB);
    }
    if (p.raw_b) p.raw_b[cell] = rawB;
    if (p.meter_b) p.meter_b[cell] = INT8 ? fminf(1.0f, rawB) : NAN;
  }
  if (RISK) {
    const int nblk = (p.S + kBlk - 1) / kBlk;
    const int S_c = p.seq_len ? p.seq_len[cell / p.Hq] : p.S;      // this cell's sequence
    const int nblk_c = (S_c + kBlk - 1) / kBlk;
    const float2* rr = p.risk_raw + (size_t)cell * p.nblk_max;
    float* ro = p.risk + (size_t)cell * p.nblk_max;
    for (int b = threadIdx.x; b < nblk; b += kMergeWarps * 32) {
      const float2 v = b < nblk_c ? rr[b] : make_float2(0.f, 0.f);
      ro[b] = (v.y == 0.f || Zt == 0.f) ? 0.f : v.y * ex2(v.x - Mx) * inv;
    }
  }
}

int seqs_per_cta_for(int scheme, int B) {
  const int cap = scheme == kBbox ? 8 : 16;
  const int n = B >= 16 ? 16 : B >= 8 ? 8 : B >= 4 ? 4 : B >= 2 ? 2 : 1;
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
