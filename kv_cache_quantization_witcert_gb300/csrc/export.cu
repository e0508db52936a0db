// Inspection kernels: unpack the fragment-ordered block store into canonical
// layouts, and expose the dither stream.  Not on the decode path.
#include "common.cuh"
#include "kernels.h"

namespace witcert {

namespace {

enum { X_KC = 0, X_VC, X_KS, X_VS, X_VZ, X_KIVI_KS, X_KIVI_KZ, X_W, X_SLOTS, X_RISK, X_VW };

__global__ void export_kernel(const ExportArgs a, size_t n) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n) return;
  const int bb = block_bytes(a.scheme);
  const int nblk = (a.S + kBlk - 1) / kBlk;
  switch (a.what) {
    case X_KC:
    case X_VC: {  // [B][S][Hkv][128]
      const int c = idx % kD, h = (idx / kD) % a.Hkv, t = (idx / ((size_t)kD * a.Hkv)) % a.S;
      const int i = idx / ((size_t)kD * a.Hkv * a.S);
      const uint8_t* bp = a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, t >> 4) * bb;
      const int r = t & 15;
      if (a.scheme == kBbox) {   // the stored bf16 values
        const int off = a.what == X_KC ? BboxLayout::KH + kbf_off(r, c) : BboxLayout::VH + vbf_off(r, c);
        reinterpret_cast<uint16_t*>(a.dst)[idx] = *reinterpret_cast<const uint16_t*>(bp + off);
        break;
      }
      uint8_t v;
      if (a.scheme == kKivi) {
        int off, bit;
        if (a.what == X_KC) kivi_k_pos(r, c, off, bit); else kivi_v_pos(r, c, off, bit);
        const uint32_t w = *reinterpret_cast<const uint32_t*>(bp + (a.what == X_KC ? KiviLayout::KC : KiviLayout::VC) + off);
        v = (uint8_t)((w >> bit) & 3u);
      } else {
        const int base = a.what == X_KC ? 0 : 2048;
        v = bp[base + (a.what == X_KC ? kcode_off(r, c) : vcode_off(r, c))];
        if (int8_layout(a.scheme)) v = (uint8_t)(v ^ 0x80u);    // stored biased by 128
      }
      reinterpret_cast<uint8_t*>(a.dst)[idx] = v;
      break;
    }
    case X_KS:
    case X_VS:
    case X_VZ: {  // [B][S][Hkv][4]
      const int G = idx % 4, h = (idx / 4) % a.Hkv, t = (idx / (4 * (size_t)a.Hkv)) % a.S;
      const int i = idx / (4 * (size_t)a.Hkv * a.S);
      const uint8_t* bp = a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, t >> 4) * bb;
      const int r = t & 15;
      __half v;
      if (a.scheme == kKivi) {
        v = reinterpret_cast<const __half*>(bp + KiviLayout::VP)[(r * 4 + G) * 2 + (a.what == X_VZ ? 1 : 0)];
      } else {
        v = a.what == X_KS ? reinterpret_cast<const __half*>(bp + Int8Layout::KS)[r * 4 + G]
                           : *reinterpret_cast<const __half*>(bp + Int8Layout::VS + vscale_off(r, G));
      }
      reinterpret_cast<__half*>(a.dst)[idx] = v;
      break;
    }
    case X_KIVI_KS:
    case X_KIVI_KZ: {  // [B][nblk][Hkv][128]
      const int c = idx % kD, h = (idx / kD) % a.Hkv, b = (idx / ((size_t)kD * a.Hkv)) % nblk;
      const int i = idx / ((size_t)kD * a.Hkv * nblk);
      const uint8_t* bp = a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, b) * bb;
      reinterpret_cast<__half*>(a.dst)[idx] =
          reinterpret_cast<const __half*>(bp + KiviLayout::KP + (a.what == X_KIVI_KZ ? 256 : 0))[kivi_kparam_idx(c)];
      break;
    }
    case X_W: {  // [B][S][Hkv][16]
      const int b = idx % kBands, h = (idx / kBands) % a.Hkv, t = (idx / ((size_t)kBands * a.Hkv)) % a.S;
      const int i = idx / ((size_t)kBands * a.Hkv * a.S);
      const uint8_t* bp = a.blocks + block_index(a.table, a.Hkv, a.nblk_max, i, h, t >> 4) * bb;
      reinterpret_cast<__half*>(a.dst)[idx] =
          *reinterpret_cast<const __half*>(bp + witness_off(a.scheme) + wit_off(t & 15, b));
      break;
    }
    case X_SLOTS: {  // [B][Hkv][nblk]
      const int b = idx % nblk;
      const size_t sh = idx / nblk;
      reinterpret_cast<int32_t*>(a.dst)[idx] = a.slots ? a.slots[sh * a.nblk_max + b] : -1;
      break;
    }
    case X_RISK: {  // [B][Hq][nblk]
      const int b = idx % nblk;
      const size_t cell = idx / nblk;
      reinterpret_cast<float*>(a.dst)[idx] = a.risk[cell * a.nblk_max + b];
      break;
    }
    case X_VW: {  // [B][S][Hkv]
      const int h = idx % a.Hkv, t = (idx / a.Hkv) % a.S;
      const int i = idx / ((size_t)a.Hkv * a.S);
      reinterpret_cast<__half*>(a.dst)[idx] = a.vwit[(((size_t)i * a.Hkv + h) * a.nblk_max + (t >> 4)) * kBlk + (t & 15)];
      break;
    }
  }
}

__global__ void dither_kernel(uint64_t seed, int layer, int kvh, int t0, int n, int tensor, float* out) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * 32) return;
  const int r = idx / 32, quad = idx % 32;
  const float4 x = dither4(seed, layer, kvh, t0 + r, quad, tensor);
  *reinterpret_cast<float4*>(out + (size_t)r * kD + 4 * quad) = x;
}

// Status of the last bounded-wait self test: 0 = satisfied, 1 = timed out.
static __device__ int g_wait_status;

// An mbarrier that expects one arrival nobody makes: the bounded wait used by the
// decode pipeline must give up after `limit_ns` and report it.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    g_wait_status = mbar_wait(smem_addr(&bar), 0, limit_ns) ? 0 : 1;
  }
}

}  // namespace

cudaError_t run_wait_selftest(uint64_t limit_ns, cudaStream_t st, int* timed_out) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(timed_out, g_wait_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e;
}

cudaError_t launch_export(const ExportArgs& a, cudaStream_t st) {
  const int nblk = (a.S + kBlk - 1) / kBlk;
  size_t n = 0;
  switch (a.what) {
    case X_KC: case X_VC: n = (size_t)a.B * a.S * a.Hkv * kD; break;
    case X_KS: case X_VS: case X_VZ: n = (size_t)a.B * a.S * a.Hkv * 4; break;
    case X_KIVI_KS: case X_KIVI_KZ: n = (size_t)a.B * nblk * a.Hkv * kD; break;
    case X_W: n = (size_t)a.B * a.S * a.Hkv * kBands; break;
    case X_SLOTS: n = (size_t)a.B * a.Hkv * nblk; break;
    case X_RISK: n = (size_t)a.B * a.Hq * nblk; break;
    case X_VW: n = (size_t)a.B * a.S * a.Hkv; break;
  }
  if (n == 0) return cudaSuccess;
  export_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a, n);
  return cudaGetLastError();
}

cudaError_t launch_dither(uint64_t seed, int layer, int kvh, int t0, int n, int tensor, float* out,
                          cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  dither_kernel<<<(n * 32 + 127) / 128, 128, 0, st>>>(seed, layer, kvh, t0, n, tensor, out);
  return cudaGetLastError();
}

}  // namespace witcert
