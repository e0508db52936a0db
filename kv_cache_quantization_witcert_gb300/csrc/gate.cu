// Meter-driven gate [WitCert summary, implementation paragraph; WitCert Lean
// page, Figure 2 and Figure 5 captions]: pick exact key blocks to page in,
// copy them from the pinned host backing store into the device pool, mark them
// repaired and zero their witnesses.
//
// Selection of one (sequence, query head) cell, a deterministic function of the
// fp32 block risks the decode reported:
//   candidates = unrepaired blocks, ranked by risk (largest first, ties to the
//   lower block index; a NaN risk counts as +inf, a risk that is not positive as 0);
//   the cell triggers if the exact sum of its candidates' risks exceeds
//   D* = sqrt(1 + 2 tau) - 1, and then takes the shortest ranked prefix whose exact
//   remaining sum is <= D*.
// "Exact" is meant literally: risks are added as integers in units of 2^-149 (every
// finite fp32 value is one), in 320-bit accumulators, and compared with floor(D* 2^149),
// so no summation order and no rounding enters a decision.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace witcert {

namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr uint32_t kInfBits = 0x7F800000u;

// ------------------------------------------------------------------ exact fixed-point sums
// A non-negative multiple of 2^-149 below 2^(320-149), as ten 32-bit limbs (little end first).
struct Big {
  uint32_t w[kBigLimbs];
};

__device__ __forceinline__ void big_zero(Big& a) {
#pragma unroll
  for (int i = 0; i < kBigLimbs; ++i) a.w[i] = 0u;
}

// a += b with one carry chain
__device__ __forceinline__ void big_add(Big& a, const Big& b) {
  asm("add.cc.u32 %0, %0, %10;\n\t"
      "addc.cc.u32 %1, %1, %11;\n\t"
      "addc.cc.u32 %2, %2, %12;\n\t"
      "addc.cc.u32 %3, %3, %13;\n\t"
      "addc.cc.u32 %4, %4, %14;\n\t"
      "addc.cc.u32 %5, %5, %15;\n\t"
      "addc.cc.u32 %6, %6, %16;\n\t"
      "addc.cc.u32 %7, %7, %17;\n\t"
      "addc.cc.u32 %8, %8, %18;\n\t"
      "addc.u32 %9, %9, %19;"
      : "+r"(a.w[0]), "+r"(a.w[1]), "+r"(a.w[2]), "+r"(a.w[3]), "+r"(a.w[4]), "+r"(a.w[5]), "+r"(a.w[6]),
        "+r"(a.w[7]), "+r"(a.w[8]), "+r"(a.w[9])
      : "r"(b.w[0]), "r"(b.w[1]), "r"(b.w[2]), "r"(b.w[3]), "r"(b.w[4]), "r"(b.w[5]), "r"(b.w[6]), "r"(b.w[7]),
        "r"(b.w[8]), "r"(b.w[9]));
}

// a += the finite, non-negative fp32 value with bit pattern `bits`: its significand M (24 bits)
// times 2^e, e = (biased exponent - 1) for normals and 0 for subnormals, in units of 2^-149.
__device__ __forceinline__ void big_add_bits(Big& a, uint32_t bits) {
  const uint32_t E = bits >> 23, mant = bits & 0x7FFFFFu;
  const uint32_t M = E ? (mant | 0x800000u) : mant;
  const uint32_t e = E ? E - 1u : 0u;
  const uint32_t q = e >> 5, sh = e & 31u;
  const uint32_t lo = M << sh, hi = sh ? (M >> (32u - sh)) : 0u;
  Big b;
#pragma unroll
  for (int i = 0; i < kBigLimbs; ++i) b.w[i] = (uint32_t)i == q ? lo : (uint32_t)i == q + 1u ? hi : 0u;
  big_add(a, b);
}

__device__ __forceinline__ bool big_gt(const Big& a, const uint32_t (&b)[kBigLimbs]) {
  bool gt = false, decided = false;
#pragma unroll
  for (int i = kBigLimbs - 1; i >= 0; --i) {
    if (!decided && a.w[i] != b[i]) {
      gt = a.w[i] > b[i];
      decided = true;
    }
  }
  return gt;
}

__device__ __forceinline__ Big big_shfl_down(const Big& a, int o) {
  Big r;
#pragma unroll
  for (int i = 0; i < kBigLimbs; ++i) r.w[i] = __shfl_down_sync(0xffffffffu, a.w[i], o);
  return r;
}

// Inclusive suffix sums over the lanes of a warp: lane l ends with the sum of lanes l..31.
__device__ __forceinline__ void big_warp_suffix(Big& a, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const Big v = big_shfl_down(a, o);
    if (lane + o < 32) big_add(a, v);
  }
}

// The rank key of a candidate: risk bits (NaN -> +inf, not positive -> 0) above the complement
// of the block index, so that descending keys are descending risk, then ascending index.
__device__ __forceinline__ unsigned long long rank_key(float r, int b) {
  const uint32_t bits = r != r ? kInfBits : (r > 0.0f ? __float_as_uint(r) : 0u);
  return ((unsigned long long)bits << 32) | (0xFFFFFFFFu - (uint32_t)b);
}
__device__ __forceinline__ uint32_t key_bits(unsigned long long k) { return (uint32_t)(k >> 32); }
__device__ __forceinline__ int key_block(unsigned long long k) { return (int)(0xFFFFFFFFu - (uint32_t)k); }

__device__ __forceinline__ unsigned long long shfl_xor64(unsigned long long v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
  return ((unsigned long long)hi << 32) | lo;
}
// Bitonic sort, descending, of the kSelThreads * P keys of a CTA.  Thread t holds positions
// t P .. t P + P - 1 in k[]: stages whose partner is in the same thread run in registers, those
// whose partner is in the same warp through shuffles, and only the others through shared
// memory (sk, element j of thread t at sk[j * kSelThreads + t], so that every access of a warp
// touches consecutive words).
template <int P>
__device__ __forceinline__ void sort_desc(unsigned long long (&k)[P], unsigned long long* sk) {
  constexpr int N = kSelThreads * P;
  const int tid = threadIdx.x;
  for (int size = 2; size <= N; size <<= 1) {
    int jj = size >> 1;
    for (; jj >= 32 * P; jj >>= 1) {
      const int tx = jj / P;                      // partner thread tid ^ tx, another warp
      __syncthreads();
#pragma unroll
      for (int j = 0; j < P; ++j) sk[j * kSelThreads + tid] = k[j];
      __syncthreads();
#pragma unroll
      for (int j = 0; j < P; ++j) {
        const unsigned long long o = sk[j * kSelThreads + (tid ^ tx)];
        const int pos = tid * P + j;
        const bool keep_max = ((pos & jj) == 0) == ((pos & size) == 0);
        k[j] = keep_max ? (k[j] > o ? k[j] : o) : (k[j] < o ? k[j] : o);
      }
    }
    for (; jj >= P; jj >>= 1) {
      const int lx = jj / P;                      // partner lane lane ^ lx
#pragma unroll
      for (int j = 0; j < P; ++j) {
        const unsigned long long o = shfl_xor64(k[j], lx);
        const int pos = tid * P + j;
        const bool keep_max = ((pos & jj) == 0) == ((pos & size) == 0);
        k[j] = keep_max ? (k[j] > o ? k[j] : o) : (k[j] < o ? k[j] : o);
      }
    }
#pragma unroll
    for (int d = P / 2; d > 0; d >>= 1) {
      if (d > jj) continue;
#pragma unroll
      for (int j = 0; j < P; ++j) {
        if (j & d) continue;
        const bool desc = ((tid * P + j) & size) == 0;
        const unsigned long long a = k[j], b = k[j | d];
        const unsigned long long mx = a > b ? a : b, mn = a > b ? b : a;
        k[j] = desc ? mx : mn;
        k[j | d] = desc ? mn : mx;
      }
    }
  }
}

// Sum of a per-thread Big over the CTA into `out` (valid in every thread afterwards).
__device__ __forceinline__ void big_block_sum(Big& a, Big (&s_w)[kSelWarps], Big& out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  big_warp_suffix(a, lane);
  if (lane == 0) s_w[warp] = a;
  __syncthreads();
  big_zero(out);
#pragma unroll 1
  for (int w = 0; w < kSelWarps; ++w) big_add(out, s_w[w]);
}

// Sum over the CTA of one float per thread, every add rounded up (so the result bounds the
// exact sum from above) or down; the same value in every thread.  s_f: kSelWarps floats.
__device__ __forceinline__ float block_sum_dir(float v, bool up, float* s_f) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = up ? __fadd_ru(v, w) : __fadd_rd(v, w);
  }
  __syncthreads();                             // earlier readers of s_f are done
  if (lane == 0) s_f[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) t = up ? __fadd_ru(t, s_f[w]) : __fadd_rd(t, s_f[w]);
  return t;
}

// Rank the n candidate keys at sk[0 .. n) (sk holds zeros from n to kSelThreads * p), take the
// shortest prefix whose exact remaining risk (the candidates' after it, plus `base`) is <= D*,
// and mark its blocks in `mask`.  Infinite risks rank first; the remaining risk before any of
// them is infinite.
template <int p>
__device__ __forceinline__ void rank_and_take(unsigned long long* sk, int n, int n_inf, const Big& base,
                                              const GateArgs& a, uint32_t* mask, Big (&s_w)[kSelWarps], int* s_count) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long k[p];
#pragma unroll
  for (int q = 0; q < p; ++q) k[q] = sk[q * kSelThreads + tid];
  sort_desc<p>(k, sk);
  // exact remaining sums: base, plus the finite risks at ranked positions after this thread's,
  // plus its own from the last position back
  Big mine;
  big_zero(mine);
#pragma unroll
  for (int q = 0; q < p; ++q)
    if (key_bits(k[q]) != kInfBits) big_add_bits(mine, key_bits(k[q]));
  Big after = mine;
  big_warp_suffix(after, lane);
  const Big next = big_shfl_down(after, 1);
  __syncthreads();                             // s_w free
  if (lane == 0) s_w[warp] = after;
  if (lane == 31) big_zero(after); else after = next;
  __syncthreads();
#pragma unroll 1
  for (int w = warp + 1; w < kSelWarps; ++w) big_add(after, s_w[w]);
  big_add(after, base);
  int cnt = 0;
#pragma unroll
  for (int q = p - 1; q >= 0; --q) {
    const int pos = tid * p + q;
    if (pos >= n) continue;
    if (pos < n_inf) { ++cnt; continue; }
    big_add_bits(after, key_bits(k[q]));
    if (big_gt(after, a.dstar)) ++cnt;
  }
  if (cnt) atomicAdd(s_count, cnt);
  __syncthreads();
  const int kstar = *s_count;                  // the remaining risk exceeds D* exactly at positions < k*
  if (kstar > 0 && tid == 0 && a.stats) atomicAdd(&a.stats[0], 1ull);
#pragma unroll
  for (int q = 0; q < p; ++q) {
    if (tid * p + q < kstar) {
      const int b = key_block(k[q]);
      atomicOr(&mask[b >> 5], 1u << (b & 31));
    }
  }
}

// One CTA per (sequence, query head) cell; up to kSelThreads * PMAX candidate blocks (the
// launch's longest sequence).  Dynamic shared memory: kSelThreads * PMAX keys.
//  1. candidates packed into shared memory, infinite risks counted;
//  2. trigger: the exact sum of the finite risks against D*, decided by sums rounded down and
//     up when they agree, exactly otherwise;
//  3. prefilter: the largest v (a 16-bit prefix of the risk bits) whose upward-rounded sum of
//     the risks below v is <= D*: no block below v can be taken, since taking every block at or
//     above v already leaves at most D*;
//  4. the blocks below v leave as an exact base sum, the others are compacted to the front;
//  5. the survivors are ranked by a sort of the smallest width that holds them.
template <int PMAX>
__global__ void __launch_bounds__(kSelThreads) gate_select_kernel(const GateArgs a) {
  extern __shared__ unsigned long long sk[];
  __shared__ Big s_w[kSelWarps];
  __shared__ float s_f[kSelWarps];
  __shared__ int s_n, s_ninf, s_count, s_warp[kSelWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cell = blockIdx.x;                 // i * Hq + j
  const int i = cell / a.Hq, j = cell % a.Hq, h = j / a.grp;
  const int nblk = ((a.seq_len ? a.seq_len[i] : a.S) + kBlk - 1) / kBlk;
  const float* risk = a.risk + (size_t)cell * a.nblk_max;
  const size_t row = ((size_t)i * a.Hkv + h) * a.nblk_max;
  if (tid == 0) { s_n = 0; s_ninf = 0; s_count = 0; }
  __syncthreads();
  // 1. candidates, packed to the front in any order
  for (int b0 = 0; b0 < nblk; b0 += kSelThreads) {
    const int b = b0 + tid;
    const bool cand = b < nblk && (a.slots ? a.slots[row + b] < 0 : !(a.repaired && a.repaired[row + b]));
    unsigned long long key = 0ull;
    if (cand) {
      key = rank_key(risk[b], b);
      if (key_bits(key) == kInfBits) atomicAdd(&s_ninf, 1);
    }
    const unsigned int ballot = __ballot_sync(0xffffffffu, cand);
    int base = 0;
    if (lane == 0 && ballot) base = atomicAdd(&s_n, __popc(ballot));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (cand) sk[base + __popc(ballot & ((1u << lane) - 1u))] = key;
  }
  __syncthreads();
  const int n = s_n, n_inf = s_ninf;
  auto finite_risk = [&](unsigned long long key) -> float {
    const uint32_t bits = key_bits(key);
    return bits == kInfBits ? 0.f : __uint_as_float(bits);
  };
  // 2. trigger
  if (n_inf == 0) {
    float up = 0.f, dn = 0.f;
    for (int m = tid; m < n; m += kSelThreads) {
      const float r = finite_risk(sk[m]);
      up = __fadd_ru(up, r);
      dn = __fadd_rd(dn, r);
    }
    const float U = block_sum_dir(up, true, s_f), L = block_sum_dir(dn, false, s_f);
    if ((double)U <= a.d_star) return;                     // exact total <= U <= D*
    if (!((double)L > a.d_star)) {                         // undecided: the exact sum decides
      Big t;
      big_zero(t);
      for (int m = tid; m < n; m += kSelThreads) big_add_bits(t, key_bits(sk[m]));
      Big total;
      big_block_sum(t, s_w, total);
      if (!big_gt(total, a.dstar)) return;
    }
  }
  // 3. prefilter: largest t in [0, 0x7F80] with RU(sum of risks whose bits < t << 16) <= D*
  int lo = 0, hi = 0x7F81;                     // t = lo is valid (an empty sum), hi is not
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    const uint32_t v = (uint32_t)mid << 16;
    float up = 0.f;
    for (int m = tid; m < n; m += kSelThreads) {
      const uint32_t bits = key_bits(sk[m]);
      if (bits < v) up = __fadd_ru(up, __uint_as_float(bits));
    }
    if ((double)block_sum_dir(up, true, s_f) <= a.d_star) lo = mid; else hi = mid;
  }
  const uint32_t v = (uint32_t)lo << 16;
  // 4. exact base of the blocks below v; the others compacted to the front, round by round
  //    (a round writes only below positions every thread has read)
  Big bs;
  big_zero(bs);
  int ns = 0;
  for (int r0 = 0; r0 < n; r0 += kSelThreads) {
    const int m = r0 + tid;
    const unsigned long long key = m < n ? sk[m] : 0ull;
    const bool keep = m < n && key_bits(key) >= v;
    if (m < n && !keep) big_add_bits(bs, key_bits(key));
    const unsigned int ballot = __ballot_sync(0xffffffffu, keep);
    __syncthreads();                           // every key of the round is read
    if (lane == 0) s_warp[warp] = __popc(ballot);
    __syncthreads();
    int off = ns;
    for (int w = 0; w < warp; ++w) off += s_warp[w];
    if (keep) sk[off + __popc(ballot & ((1u << lane) - 1u))] = key;
    for (int w = 0; w < kSelWarps; ++w) ns += s_warp[w];
  }
  Big base;
  big_block_sum(bs, s_w, base);
  // 5. rank the survivors with the narrowest sort that holds them
  int pp = 1;
  while (kSelThreads * pp < ns) pp <<= 1;
  for (int m = ns + tid; m < kSelThreads * pp; m += kSelThreads) sk[m] = 0ull;
  __syncthreads();
  uint32_t* mask = a.selmask + ((size_t)i * a.Hkv + h) * (a.nblk_max / 32 + 1);
  if (pp == 1) rank_and_take<1>(sk, ns, n_inf, base, a, mask, s_w, &s_count);
  else if (pp == 2) { if constexpr (PMAX >= 2) rank_and_take<2>(sk, ns, n_inf, base, a, mask, s_w, &s_count); }
  else if (pp == 4) { if constexpr (PMAX >= 4) rank_and_take<4>(sk, ns, n_inf, base, a, mask, s_w, &s_count); }
  else if (pp == 8) { if constexpr (PMAX >= 8) rank_and_take<8>(sk, ns, n_inf, base, a, mask, s_w, &s_count); }
  else if (pp == 16) { if constexpr (PMAX >= 16) rank_and_take<16>(sk, ns, n_inf, base, a, mask, s_w, &s_count); }
  else { if constexpr (PMAX >= 32) rank_and_take<32>(sk, ns, n_inf, base, a, mask, s_w, &s_count); }
}

// Per (sequence, KV head), one warp: turn the selection bitmap into pool slots and todo
// entries, 32 bitmap words at a time (one pool and one todo reservation per batch).
// A selected block is unrepaired (the selection ranks unrepaired blocks only); slots past
// the pool's capacity are counted as dropped.
__global__ void __launch_bounds__(128) gate_compact_kernel(const GateArgs a) {
  const int sh = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (sh >= a.B * a.Hkv) return;
  const int nwords = a.nblk_max / 32 + 1;
  uint32_t* mask = a.selmask + (size_t)sh * nwords;
  const unsigned int cap = (unsigned int)a.pool_capacity;
  for (int w0 = 0; w0 < nwords; w0 += 32) {
    const int w = w0 + lane;
    uint32_t bits = w < nwords ? mask[w] : 0u;
    if (bits) mask[w] = 0u;
    const int cnt = __popc(bits);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const unsigned int total = (unsigned int)__shfl_sync(0xffffffffu, incl, 31);
    if (total == 0) continue;
    unsigned int base = 0, tbase = 0, fit = 0;
    if (lane == 0) {
      base = atomicAdd(a.pool_next, total);
      fit = base >= cap ? 0u : min(total, cap - base);
      atomicAdd(&a.stats[1], (unsigned long long)total);
      if (fit < total) atomicAdd(&a.stats[4], (unsigned long long)(total - fit));
      if (fit) tbase = atomicAdd(a.todo_count, fit);
    }
    base = __shfl_sync(0xffffffffu, base, 0);
    fit = __shfl_sync(0xffffffffu, fit, 0);
    tbase = __shfl_sync(0xffffffffu, tbase, 0);
    unsigned int r = (unsigned int)(incl - cnt);
    while (bits) {
      const int b = w * 32 + __ffs(bits) - 1;
      bits &= bits - 1;
      if (r < fit) a.todo[tbase + r] = make_int4(sh / a.Hkv, sh % a.Hkv, b, (int)(base + r));
      ++r;
    }
  }
}

// Copy each todo block (16 exact key rows) from mapped host memory, then publish it.
__global__ void __launch_bounds__(256) gate_pagein_kernel(const GateArgs a) {
  const unsigned int n = *a.todo_count;
  const int row_bytes = kD * a.elem_bytes;
  const int blk_bytes = kBlk * row_bytes;
  for (unsigned int e = blockIdx.x; e < n; e += gridDim.x) {
    const int4 td = a.todo[e];
    const int i = td.x, h = td.y, b = td.z, slot = td.w;
    const size_t sh = (size_t)i * a.Hkv + h;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(a.backing) + (sh * a.backing_rows + (size_t)b * kBlk) * row_bytes;
    uint8_t* dst = reinterpret_cast<uint8_t*>(a.pool) + (size_t)slot * blk_bytes;
    for (int k = threadIdx.x * 16; k < blk_bytes; k += blockDim.x * 16)
      *reinterpret_cast<uint4*>(dst + k) = *reinterpret_cast<const uint4*>(src + k);
    __syncthreads();
    if (threadIdx.x < 32) {
      uint8_t* wreg = a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, b) * block_bytes(a.scheme) +
                      witness_off(a.scheme);
      reinterpret_cast<uint4*>(wreg)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    }
    __threadfence();
    if (threadIdx.x == 0) {
      a.slots[sh * a.nblk_max + b] = slot;
      atomicAdd(&a.stats[2], 1ull);
      atomicAdd(&a.stats[3], (unsigned long long)blk_bytes);
    }
    __syncthreads();
  }
}

template <int P>
cudaError_t launch_select(const GateArgs& a, cudaStream_t st) {
  const int smem = kSelThreads * P * (int)sizeof(unsigned long long);
  cudaError_t e = cudaFuncSetAttribute(gate_select_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  gate_select_kernel<P><<<a.B * a.Hq, kSelThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

// floor(d 2^149) as limbs: d is a float64 >= 0 below 2^170 (D* of a float tau is below 2^65).
void fixed_limbs(double d, uint32_t (&w)[kBigLimbs]) {
  for (int i = 0; i < kBigLimbs; ++i) w[i] = 0u;
  if (!(d > 0.0)) return;
  int ex = 0;
  const double f = std::frexp(d, &ex);                       // d = f 2^ex, f in [1/2, 1)
  const unsigned long long m = (unsigned long long)std::ldexp(f, 53);   // exact 53-bit integer
  for (int b = 0; b < 53; ++b) {
    if (!((m >> b) & 1ull)) continue;
    const int pos = b + ex - 53 + 149;                       // bit position in units of 2^-149
    if (pos >= 0 && pos < 32 * kBigLimbs) w[pos >> 5] |= 1u << (pos & 31);
  }
}

int gate_max_blocks() { return kSelThreads * kSelMaxKeysPerThread; }

cudaError_t launch_gate_select(const GateArgs& a0, cudaStream_t st) {
  GateArgs a = a0;
  fixed_limbs(a.d_star, a.dstar);
  const int nblk = (a.S + kBlk - 1) / kBlk;
  if (nblk > gate_max_blocks()) return cudaErrorInvalidValue;
  int P = 1;
  while (kSelThreads * P < nblk) P <<= 1;
  switch (P) {
    case 1: return launch_select<1>(a, st);
    case 2: return launch_select<2>(a, st);
    case 4: return launch_select<4>(a, st);
    case 8: return launch_select<8>(a, st);
    case 16: return launch_select<16>(a, st);
    default: return launch_select<32>(a, st);
  }
}

cudaError_t launch_gate(const GateArgs& a, cudaStream_t st) {
  cudaError_t e = launch_gate_select(a, st);
  if (e != cudaSuccess) return e;
  gate_compact_kernel<<<(a.B * a.Hkv * 32 + 127) / 128, 128, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gate_pagein_kernel<<<1024, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace witcert
