// Internal kernel launchers (host side).  Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace witcert {

// Split record: m (log2 units), Z, S_A, S_B, S_V, three unused, acc[128]
constexpr int kPartStride = 136;
constexpr int kPartAcc = 8;

struct WriteArgs {
  uint8_t* blocks;           // layer base: [B][Hkv][nblk_max][block_bytes], or the layer's page pool
  const int32_t* table;      // paged store: [B][nblk_max] page of each block (shared by layers), or null
  int nblk_max;
  const void* K;             // [B][n_tok][Hkv][128]
  const void* V;
  const void* Kh;            // black-box scheme: the tensor function's outputs, same layout as K, V
  const void* Vh;
  __half* vwit;              // layer base [B][Hkv][nblk_max][16] value witnesses, or null
  int B, Hkv, n_tok, t0, layer, backing_rows;   // backing_rows: rows per (seq, KV head) in the backing store
  int tok_begin, tok_count;  // tokens of this write a per-token launch covers
  int pos0;                  // global position of the cache's first token (dither key)
  int is_bf16;
  int late_wait;             // token, block and KIVI value kernels wait for their predecessor at
                             // their end instead of their start (see ChainEntry in write.cu)
  uint64_t seed;
  uint32_t rk0[10], rk1[10]; // Philox round keys of `seed` (as in DecodeArgs)
  void* backing;             // device-mapped pinned host, layer base [B][Hkv][backing_rows][128], or null
  const int32_t* slots;      // layer base [B][Hkv][nblk_max], or null
  void* pool;                // exact-key pool [slots][16][128]
  float* kivi_tail;          // layer base [B][Hkv][16][128] (KIVI)
  unsigned long long* clamps;
};

struct DecodeArgs {
  const uint8_t* blocks;     // layer base (contiguous store or page pool)
  const int32_t* table;      // paged store: [B][nblk_max] pages, or null
  int nblk_max;
  const int32_t* slots;      // layer base or null
  const void* pool;
  const float* kivi_tail;    // layer base (KIVI)
  const void* q;             // [B][Hq][128]
  int is_bf16;
  int B, Hq, Hkv, grp, S, n_splits, seqs_per_cta;   // S: the longest sequence's length
  const int* seq_len;        // [B] per-sequence lengths of a ragged batch (device), or null (all S)
  double log2dl;             // ln(2 / delta_loc): Tier B's kappa per sequence when seq_len is set
  int dirty_blk;             // first block the immediately preceding kernel may write (INT_MAX: none)
  uint64_t seed;
  uint32_t rk0[10], rk1[10]; // Philox round keys of `seed` (key words advanced by the Weyl increments)
  int layer;
  float kappa;               // sqrt(2 ln(2S/delta_loc)), rounded up (Tier B)
  float* part;               // [B][Hq][n_splits][kPartStride]
  float2* risk_raw;          // [B][Hq][nblk_max] (block max in log2 units, risk sum), or null
  float* risk;               // [B][Hq][nblk_max] normalized block risk, or null
  float* out;                // [B][Hq][128]
  float *meter_a, *meter_b, *raw_a, *raw_b;
  const __half* vwit;        // layer base [B][Hkv][nblk_max][16] value witnesses, or null
  float* meter_v;            // [B][Hq] value meter, or null
  int* err;                  // device error word (spin limits)
  const uint8_t* next_blocks;  // the next layer's base: its first blocks are prefetched into L2, or null
  int pos0;                  // global position of the cache's first token (dither key)
  float* part_out;           // [B][Hq][kPartStride]: merge writes each cell's combined record here
                             // (context-parallel shard) instead of the output and meters, or null
  bool meter;
};

// Sequences of one ragged append launch, passed by value: sequence seq[k] appends the
// off[k+1] - off[k] tokens that start at packed input row row0[k] (inputs [rows][Hkv][128]),
// at positions t0[k], t0[k] + 1, ...; off is the launch's running token count.
constexpr int kRaggedPerLaunch = 128;
struct RaggedArgs {
  int n_seq;
  int seq[kRaggedPerLaunch], t0[kRaggedPerLaunch], row0[kRaggedPerLaunch], off[kRaggedPerLaunch + 1];
};
// New per-sequence lengths, up to kRaggedPerLaunch of them: dst[idx[k]] = len[k] (idx indexes
// the [layer][sequence] array).
struct LengthArgs {
  int* dst;
  int n;
  int idx[kRaggedPerLaunch], len[kRaggedPerLaunch];
};

// pdl: launch with programmatic stream serialization (off right after an event wait).
cudaError_t launch_write(int scheme, const WriteArgs& a, cudaStream_t st, bool pdl);
// Ragged appends of the sequences in g (KIVI: values and the key backing store only).
cudaError_t launch_write_ragged(int scheme, const WriteArgs& a, const RaggedArgs& g, cudaStream_t st, bool pdl);
cudaError_t launch_set_lengths(const LengthArgs& u, cudaStream_t st, bool pdl);
// KIVI key blocks a (uniform) write completes, then its unfinished block's exact tail.
cudaError_t launch_kivi_keys(const WriteArgs& a, cudaStream_t st, bool pdl);
// Philox4x32-10 round keys of a 64-bit seed: key (seed mod 2^32, seed div 2^32) advanced
// by 0x9E3779B9 / 0xBB67AE85 before every round but the first.
void philox_round_keys(uint64_t seed, uint32_t (&rk0)[10], uint32_t (&rk1)[10]);
// Split-KV decode + merge.  Returns the split kernel's launch error; `split_start`
// and `split_stop` (optional) bracket the split kernel alone.
cudaError_t launch_decode(int scheme, const DecodeArgs& a, int sm_count, cudaStream_t st,
                          cudaEvent_t split_start, cudaEvent_t split_stop, bool pdl);
int decode_ctas_per_sm(int scheme, const DecodeArgs& a);
// Merge kernel alone over caller-given records a.part [B][Hq][a.n_splits][kPartStride].
cudaError_t launch_merge_records(int scheme, const DecodeArgs& a, cudaStream_t st);
int decode_auto_splits(int scheme, int B, int Hkv, int nblk, int sm_count, int per_sm);
// Device address (current device) and size of the library's static split scratch,
// used by witcert_decode_noalloc; the first call on a device looks the address up.
cudaError_t decode_static_scratch(float** ptr, size_t* bytes);

// Exact fixed-point sums of the gate: 320 bits in units of 2^-149 (ten 32-bit limbs).
constexpr int kBigLimbs = 10;
// Keys a selection CTA sorts per thread, at most; with 512 threads the gate ranks up to
// 16384 blocks (262144 tokens) per sequence.
constexpr int kSelMaxKeysPerThread = 32;

struct GateArgs {
  const float* risk;         // [B][Hq][nblk_max] (this layer)
  int32_t* slots;            // [B][Hkv][nblk_max] (this layer), or null: candidacy from `repaired`
  const uint8_t* repaired;   // [B][Hkv][nblk_max] nonzero = not a candidate (used when slots is null), or null
  uint32_t* selmask;         // [B][Hkv][nblk_max/32 + 1] scratch bitmap
  int4* todo;                // [capacity] (seq, kv head, block, slot)
  unsigned int* todo_count;  // device counter (reset per call)
  unsigned int* pool_next;   // device counter (persistent)
  unsigned long long* stats; // [6] device counters (witcert_gate_stats order)
  uint8_t* blocks;           // layer base (contiguous store or page pool)
  const int32_t* table;      // paged store: [B][nblk_max] pages, or null
  const void* backing;       // device-mapped pinned host, layer base
  void* pool;
  int nblk_max, B, Hq, Hkv, grp, S, backing_rows, pool_capacity, scheme, elem_bytes;
  const int* seq_len;        // [B] per-sequence lengths (ragged batch), or null (all S)
  double d_star;             // sqrt(1 + 2 tau) - 1 in float64
  uint32_t dstar[kBigLimbs]; // floor(d_star 2^149), filled by the launcher
};
// Selection, bitmap compaction and page-in of one layer.
cudaError_t launch_gate(const GateArgs& a, cudaStream_t st);
// Selection alone: sets the bits of a.selmask ([B][Hkv][nblk_max/32 + 1], zeroed by the caller)
// of the blocks the cells ask for; a.stats may be null.  Fails for more than gate_max_blocks().
cudaError_t launch_gate_select(const GateArgs& a, cudaStream_t st);
int gate_max_blocks();
void fixed_limbs(double d, uint32_t (&w)[kBigLimbs]);

struct ExportArgs {
  const uint8_t* blocks;
  const int32_t* table;      // paged store, or null
  int nblk_max, B, Hkv, Hq, S, scheme;
  const int32_t* slots;
  const float* risk;
  const __half* vwit;        // layer base [B][Hkv][nblk_max][16], or null
  void* dst;
  int what;
};
cudaError_t launch_export(const ExportArgs& a, cudaStream_t st);
// Runs the bounded mbarrier wait against a barrier nothing completes; sets *timed_out.
cudaError_t run_wait_selftest(uint64_t limit_ns, cudaStream_t st, int* timed_out);
cudaError_t launch_dither(uint64_t seed, int layer, int kvh, int t0, int n, int tensor, float* out,
                          cudaStream_t st);
// Writers' quotient x / s (reciprocal and one correction) against the IEEE quotient, for every
// positive fp16 scale s and every bf16 x with |x| <= 127.5 s plus n_f32 seeded fp32 x per
// scale; *mismatches counts the pairs that differ (synchronous).
cudaError_t run_quotient_selftest(int n_f32, uint64_t seed, unsigned long long* mismatches, cudaStream_t st);

}  // namespace witcert
