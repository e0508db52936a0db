// Meter-driven gate [WitCert summary, implementation paragraph; WitCert Lean
// page, Figure 2 and Figure 5 captions]: pick exact key blocks to page in,
// copy them from the pinned host backing store into the device pool, mark them
// repaired and zero their witnesses.
//
// Selection of one (sequence, query head) cell, a deterministic function of the
// fp32 block risks the decode reported:
//   candidates = unrepaired blocks, ordered by risk (largest first, ties to the
//   lower block index); remaining-risk sums in fp64 in a fixed order: runs of 32
//   ranked blocks each summed from the run's last block upward (one thread per
//   run), run totals summed from the last run upward, and the remaining risk
//   after block j = j's run-local sum + the runs after it; the cell triggers if
//   the full sum exceeds D* = sqrt(1 + 2 tau) - 1 and then takes the shortest
//   prefix whose remaining sum is <= D*.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace witcert {

namespace {

constexpr int kSelThreads = 512;
constexpr int kRun = 32;

__device__ __forceinline__ double key_risk(unsigned long long key) {
  return (double)__uint_as_float(~(unsigned int)(key >> 32));
}

// Dynamic shared memory: keys [npow2] u64, run-local sums [npow2] f64, runs after [npow2/32] f64.
__global__ void __launch_bounds__(kSelThreads) gate_select_kernel(const GateArgs a, int npow2) {
  extern __shared__ unsigned long long keys[];
  double* local = reinterpret_cast<double*>(keys + npow2);
  double* after = local + npow2;
  __shared__ double red[kSelThreads];
  __shared__ int s_n, s_jmax;
  const int cell = blockIdx.x;                 // i * Hq + j
  const int i = cell / a.Hq, j = cell % a.Hq, h = j / a.grp;
  const int nblk = ((a.seq_len ? a.seq_len[i] : a.S) + kBlk - 1) / kBlk;
  const float* risk = a.risk + (size_t)cell * a.nblk_max;
  const int32_t* slots = a.slots + ((size_t)i * a.Hkv + h) * a.nblk_max;
  if (threadIdx.x == 0) { s_n = 0; s_jmax = -1; }
  __syncthreads();
  // the cell's candidate keys, packed to the front in any order (the sort ranks them), so the
  // sort covers the next power of two above the candidates rather than above the blocks
  double part = 0.0;
  const int lane = threadIdx.x & 31;
  for (int b0 = 0; b0 < nblk; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    const bool cand = b < nblk && slots[b] < 0;
    unsigned long long key = 0ull;
    if (cand) {
      const float r = risk[b];
      part += (double)r;
      key = ((unsigned long long)(~__float_as_uint(r)) << 32) | (unsigned int)b;
    }
    const unsigned int ballot = __ballot_sync(0xffffffffu, cand);
    int base = 0;
    if (lane == 0 && ballot) base = atomicAdd(&s_n, __popc(ballot));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (cand) keys[base + __popc(ballot & ((1u << lane) - 1u))] = key;
  }
  red[threadIdx.x] = part;
  __syncthreads();
  const int n = s_n;
  int npc = 1;
  while (npc < n) npc <<= 1;                   // <= npow2: n <= nblk
  for (int k = n + threadIdx.x; k < npc; k += blockDim.x) keys[k] = ~0ull;
  for (int s = blockDim.x / 2; s; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  // a parallel sum differs from the run-ordered one by far less than 1e-9 relative:
  // cells clearly below D* skip the ordered sums
  if (red[0] <= a.d_star * (1.0 - 1e-9)) return;
  // bitonic sort, ascending keys = descending risk then ascending block; each thread
  // takes compare-exchange pairs (x, x + jj) directly, x having bit jj clear
  for (int k = 2; k <= npc; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int pr = threadIdx.x; pr < (npc >> 1); pr += blockDim.x) {
        const int x = ((pr & ~(jj - 1)) << 1) | (pr & (jj - 1)), y = x + jj;
        const unsigned long long kx = keys[x], ky = keys[y];
        const bool up = (x & k) == 0;
        if ((kx > ky) == up) { keys[x] = ky; keys[y] = kx; }
      }
      __syncthreads();
    }
  }
  // run-local remaining sums, one thread per run of kRun ranked blocks
  const int nruns = (n + kRun - 1) / kRun;
  for (int rr = threadIdx.x; rr < nruns; rr += blockDim.x) {
    const int lo = rr * kRun, hi = min(n, lo + kRun);
    double s = 0.0;
    for (int m = hi - 1; m >= lo; --m) {
      s = s + key_risk(keys[m]);
      local[m] = s;
    }
    after[rr] = s;                 // run total for now
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double u = 0.0;
    for (int rr = nruns - 1; rr >= 0; --rr) {
      const double tot = after[rr];
      after[rr] = u;
      u = u + tot;
    }
  }
  __syncthreads();
  // the remaining sums never increase down the list: the cut is one past the last one above D*
  int jmax = -1;
  for (int m = threadIdx.x; m < n; m += blockDim.x)
    if (local[m] + after[m / kRun] > a.d_star) jmax = m;
  if (jmax >= 0) atomicMax(&s_jmax, jmax);
  __syncthreads();
  const int kstar = s_jmax + 1;
  if (kstar > 0 && threadIdx.x == 0) atomicAdd(&a.stats[0], 1ull);
  uint32_t* mask = a.selmask + ((size_t)i * a.Hkv + h) * (a.nblk_max / 32 + 1);
  for (int m = threadIdx.x; m < kstar; m += blockDim.x) {
    const int b = (int)(keys[m] & 0xFFFFFFFFu);
    atomicOr(&mask[b >> 5], 1u << (b & 31));
  }
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

}  // namespace

cudaError_t launch_gate(const GateArgs& a, cudaStream_t st) {
  const int nblk = (a.S + kBlk - 1) / kBlk;
  int npow2 = 1;
  while (npow2 < nblk) npow2 <<= 1;
  const size_t smem = (size_t)npow2 * (sizeof(unsigned long long) + sizeof(double)) +
                      (size_t)(npow2 / kRun + 1) * sizeof(double);
  cudaError_t e = cudaFuncSetAttribute(gate_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gate_select_kernel<<<a.B * a.Hq, kSelThreads, smem, st>>>(a, npow2);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gate_compact_kernel<<<(a.B * a.Hkv * 32 + 127) / 128, 128, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gate_pagein_kernel<<<1024, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace witcert
