// Meter-driven gate [WitCert summary, implementation paragraph; WitCert Lean
// page, Figure 2 and Figure 5 captions]: pick exact key blocks to page in,
// copy them from the pinned host backing store into the device pool, mark them
// repaired and zero their witnesses.
//
// Selection of one (sequence, query head) cell, a deterministic function of the
// fp32 block risks the decode reported:
//   candidates = unrepaired blocks, ordered by risk (largest first, ties to the
//   lower block index); suffix sums of that order accumulated in fp64 from the
//   last candidate upward; the cell triggers if the full sum exceeds
//   D* = sqrt(1 + 2 tau) - 1 and then takes the shortest prefix whose
//   remaining suffix is <= D*.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace witcert {

namespace {

constexpr int kSelThreads = 256;

__global__ void __launch_bounds__(kSelThreads) gate_select_kernel(const GateArgs a, int npow2) {
  extern __shared__ unsigned long long keys[];
  __shared__ double red[kSelThreads];
  __shared__ int kstar;
  const int cell = blockIdx.x;                 // i * Hq + j
  const int i = cell / a.Hq, j = cell % a.Hq, h = j / a.grp;
  const int nblk = (a.S + kBlk - 1) / kBlk;
  const float* risk = a.risk + (size_t)cell * a.nblk_max;
  const int32_t* slots = a.slots + ((size_t)i * a.Hkv + h) * a.nblk_max;
  double part = 0.0;
  for (int b = threadIdx.x; b < npow2; b += blockDim.x) {
    unsigned long long key = ~0ull;
    if (b < nblk && slots[b] < 0) {
      const float r = risk[b];
      part += (double)r;
      key = ((unsigned long long)(~__float_as_uint(r)) << 32) | (unsigned int)b;
    }
    keys[b] = key;
  }
  red[threadIdx.x] = part;
  __syncthreads();
  for (int s = blockDim.x / 2; s; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  // a parallel sum differs from the ordered one by far less than 1e-9 relative:
  // cells clearly below D* skip the exact walk
  if (red[0] <= a.d_star * (1.0 - 1e-9)) return;
  // bitonic sort, ascending keys = descending risk then ascending block
  for (int k = 2; k <= npow2; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int x = threadIdx.x; x < npow2; x += blockDim.x) {
        const int y = x ^ jj;
        if (y > x) {
          const unsigned long long kx = keys[x], ky = keys[y];
          const bool up = (x & k) == 0;
          if ((kx > ky) == up) { keys[x] = ky; keys[y] = kx; }
        }
      }
      __syncthreads();
    }
  }
  if (threadIdx.x == 0) {
    int n = 0;
    while (n < npow2 && keys[n] != ~0ull) ++n;
    double suffix = 0.0;
    int k = n;
    while (k > 0) {
      const double s_new = suffix + (double)__uint_as_float(~(unsigned int)(keys[k - 1] >> 32));
      if (s_new > a.d_star) break;
      suffix = s_new;
      --k;
    }
    kstar = k;
    if (k > 0) atomicAdd(&a.stats[0], 1ull);
  }
  __syncthreads();
  uint32_t* mask = a.selmask + ((size_t)i * a.Hkv + h) * (a.nblk_max / 32 + 1);
  for (int m = threadIdx.x; m < kstar; m += blockDim.x) {
    const int b = (int)(keys[m] & 0xFFFFFFFFu);
    atomicOr(&mask[b >> 5], 1u << (b & 31));
  }
}

// Per (sequence, KV head): turn the selection bitmap into pool slots and a todo list.
__global__ void gate_compact_kernel(const GateArgs a) {
  const int sh = blockIdx.x * blockDim.x + threadIdx.x;
  if (sh >= a.B * a.Hkv) return;
  const int nwords = a.nblk_max / 32 + 1;
  uint32_t* mask = a.selmask + (size_t)sh * nwords;
  const int32_t* slots = a.slots + (size_t)sh * a.nblk_max;
  for (int w = 0; w < nwords; ++w) {
    uint32_t bits = mask[w];
    mask[w] = 0u;
    while (bits) {
      const int b = w * 32 + __ffs(bits) - 1;
      bits &= bits - 1;
      if (slots[b] >= 0) continue;
      atomicAdd(&a.stats[1], 1ull);
      const unsigned int slot = atomicAdd(a.pool_next, 1u);
      if ((int)slot >= a.pool_capacity) { atomicAdd(&a.stats[4], 1ull); continue; }
      const unsigned int e = atomicAdd(a.todo_count, 1u);
      a.todo[e] = make_int4(sh / a.Hkv, sh % a.Hkv, b, (int)slot);
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
      uint8_t* wreg = a.blocks + ((sh * a.nblk_max) + b) * block_bytes(a.scheme) + witness_off(a.scheme);
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
  const size_t smem = (size_t)npow2 * sizeof(unsigned long long);
  cudaError_t e = cudaFuncSetAttribute(gate_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gate_select_kernel<<<a.B * a.Hq, kSelThreads, smem, st>>>(a, npow2);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gate_compact_kernel<<<(a.B * a.Hkv + 127) / 128, 128, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gate_pagein_kernel<<<1024, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace witcert
