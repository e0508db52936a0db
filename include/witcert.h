/*
 * witcert.h — C ABI of the GB300 metered KV-cache decode library.
 *
 * The method is WitCert ("WitCert: Sound Runtime Risk Observability and Gating
 * for KV-Cache Quantization").  Citations below name its pages:
 *   [summary]   technical summary page: witness paragraph with Lemma 1,
 *               Theorem 2, the Tier B paragraph, the implementation
 *               paragraph, the closing improvements list (TV bound);
 *   [Lean page] paperswithlean.com page: Approach, Figure 2 and Figure 5;
 *   [abstract]  arXiv abstract: the meter is sound for any cache-preserving
 *               black-box quantizer, and any scheme given as one tensor
 *               function is measured.
 *
 * Conventions for every call:
 *   - Pointers documented as "device" must be CUDA device pointers (or managed
 *     memory) on the device that was current when the cache was created;
 *     "host" pointers are ordinary host memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls are asynchronous on that stream unless stated otherwise.
 *   - The caller owns all buffers it passes; the cache owns its own device
 *     pools, its pinned host backing store and its internal side stream.
 *   - Errors are returned as witcert_status codes; nothing throws across the
 *     ABI.  witcert_last_error() gives a thread-local message for the last
 *     failing call on the calling thread.
 *   - A cache is used from one host thread at a time.
 *   - head_dim is 128; the KV-head group size Hq/Hkv is at most 8.
 */
#ifndef WITCERT_H
#define WITCERT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WITCERT_OK = 0,
  WITCERT_EINVAL = -1,     /* bad argument or configuration */
  WITCERT_ENOMEM = -2,     /* device or pinned host allocation failed */
  WITCERT_ECUDA = -3,      /* a CUDA runtime call or kernel launch failed */
  WITCERT_ETIMEDOUT = -4,  /* a bounded wait ran out (host deadline or device spin limit) */
  WITCERT_EPAGEIN = -5,    /* gate page-in could not complete (pool exhausted, injected fault) */
  WITCERT_ESTATE = -6      /* call not valid in the cache's current state */
} witcert_status;

typedef enum {
  WITCERT_INT8_DITHER = 0, /* subtractively dithered INT8, per-(token, 32-channel) fp16 scales [summary, Tier B] */
  WITCERT_FP8_E4M3 = 1,    /* black-box raw cast to OCP E4M3, no scale [summary, gate results] */
  WITCERT_KIVI2 = 2,       /* KIVI-style asymmetric 2-bit: K per channel over 16 tokens, V per token per 32 channels */
  WITCERT_INT8_RTN = 3,    /* INT8 with the same scales, rounded to nearest without dither (the dithered
                              quantizer with xi = 0); Tier A only */
  WITCERT_BLACKBOX = 4     /* any tensor function f [abstract]: the caller passes f(K), f(V) with every
                              write (witcert_write_hat); the cache keeps them as bfloat16 (544 B per token
                              and KV head with the witness); Tier A only */
} witcert_scheme;

typedef enum {
  WITCERT_F32 = 0,         /* float32 K, V and q */
  WITCERT_BF16 = 1         /* bfloat16 K, V and q */
} witcert_dtype;

typedef struct {
  int n_layers;            /* L in delta_loc = delta_req / (L*H*T) */
  int n_q_heads;           /* Hq (H in delta_loc) */
  int n_kv_heads;          /* Hkv; Hq must be a multiple, Hq/Hkv <= 8 */
  int head_dim;            /* must be 128 */
  int batch;               /* sequences held by the cache; each has its own length per layer */
  int max_tokens;          /* capacity per sequence per layer */
  witcert_scheme scheme;   /* fixed for the cache's lifetime */
  witcert_dtype kv_dtype;  /* dtype of K, V and q passed to write/decode, and of the backing store */
  uint64_t seed;           /* Philox key of the dither stream (INT8 scheme) */
  int total_steps;         /* T in delta_loc: decode steps per request */
  int n_splits;            /* KV splits per (sequence, KV head) in decode; 0 = choose from the SM count */
  int max_repair_blocks;   /* capacity of the exact-key pool in 16-token blocks; 0 disables the gate
                              and the pinned backing store */
  int pos_offset;          /* global position of the cache's first token: a cache holding one slice of
                              a longer context (one shard of a context-parallel decode) keys its dither
                              on global positions; 0 for a whole context */
  int v_witness;           /* nonzero: also keep the value witness wv_t >= ||v_t - v^_t|| (whole row,
                              fp16 rounded up; 2 B per token and KV head) and report the value meter
                              E_V = sum_t p~_t wv_t, which bounds || sum_t p~_t (v_t - v^_t) || by the
                              triangle inequality.  The pages define no value-side bound: this is the
                              value counterpart of the key witness, a reading of this library. */
  int max_pages;           /* > 0: paged block store.  Each layer holds a pool of max_pages pages, a page
                              being one 16-token block of every KV head of one sequence; a per-sequence
                              page table (shared by the layers) maps a sequence's blocks to pages, taken
                              as writes reach new blocks and given back by witcert_reset_sequence, so
                              sequences of different lengths share the pool instead of each reserving
                              max_tokens.  max_tokens stays the per-sequence cap.  bf16 caches only.
                              0: every sequence owns max_tokens of contiguous blocks. */
} witcert_config;

typedef struct witcert_cache witcert_cache;

typedef struct {
  uint64_t cells_triggered;   /* (sequence, query head) cells whose meter exceeded tau */
  uint64_t blocks_selected;   /* distinct (layer, sequence, KV head, block) picked for repair */
  uint64_t blocks_paged_in;   /* blocks copied from the backing store into the exact pool */
  uint64_t bytes_paged_in;    /* host-to-device bytes moved by page-in */
  uint64_t blocks_dropped;    /* selected but not repaired because the pool was full */
  uint64_t gate_calls;
} witcert_gate_counters;

typedef struct {
  uint64_t tokens_written;    /* token x KV head rows written, all layers */
  uint64_t decode_calls;
  uint64_t int8_clamps;       /* INT8 codes clamped to [-128, 127] (expected 0) */
  uint64_t device_errors;     /* spin limits hit inside kernels (expected 0) */
  double decode_kernel_ms;    /* summed split-kernel time while profiling is on */
  uint64_t decode_kernel_launches;
  int last_n_splits;          /* KV splits used by the most recent decode */
  uint64_t pages_used;        /* paged store: pages held by sequences (0 for a contiguous store) */
} witcert_stats_t;

/* Create a cache.  Allocates the compressed store, the witness store, the
 * split scratch and, when max_repair_blocks > 0, the exact-key pool and a
 * pinned, device-mapped host backing store of exact keys.  Memory is zeroed.
 * Synchronous.  Returns EINVAL for unsupported shapes (among them a cache with the gate
 * enabled and max_tokens above 262144: the gate ranks at most 16384 blocks of a sequence),
 * ENOMEM on allocation failure (nothing is leaked). */
witcert_status witcert_create(const witcert_config* cfg, witcert_cache** out);

/* Free everything the cache owns.  Synchronizes the device first. */
witcert_status witcert_destroy(witcert_cache* cache);

/* Write path [summary, implementation paragraph (the write side keeps a
 * witness per token and head); Tier B paragraph for the dithered quantizer;
 * witness paragraph for w_{t,b} = ||r_{t,b}||].  Appends n_tok tokens to every sequence of
 * `layer` at positions len..len+n_tok-1, where len is the layer's current
 * length.  K and V are device arrays [batch][n_tok][n_kv_heads][128] of
 * kv_dtype, contiguous; keys are post-RoPE.  Stores codes and scales, and the
 * key witness of 16 bands (band b = dims 4b..4b+3 and 64+4b..64+4b+3, whole
 * RoPE pairs of the rotate-half layout) as fp16 rounded up.  With the gate
 * enabled it also writes the exact keys into the pinned backing store.
 * EINVAL if layer is out of range or the capacity would be exceeded. */
witcert_status witcert_write(witcert_cache* cache, int layer, const void* K, const void* V,
                             int n_tok, void* stream);

/* Write path of the black-box scheme [abstract: any scheme registered as one tensor
 * function is measured; Tier A holds for any cache-preserving black-box quantizer].
 * K, V as in witcert_write; K_hat, V_hat are the tensor function's outputs f(K), f(V)
 * in the same layout and dtype.  The cache stores bf16(K_hat), bf16(V_hat) (nearest
 * even; unchanged for bf16 inputs), and the key witness w_{t,b} = ||K - bf16(K_hat)||
 * of each band, so the decode and the bound use exactly what is stored.  K_hat and V_hat
 * must be finite: the rows of a sequence's last block past its length take part in the
 * decode's P.V product with weight 0, and a non-finite value left there (by the rows'
 * occupant before a reset, or in a page that held another sequence) makes 0 x inf a NaN in
 * that later sequence's output.  EINVAL on a cache of another scheme (which takes
 * witcert_write) and as witcert_write otherwise. */
witcert_status witcert_write_hat(witcert_cache* cache, int layer, const void* K, const void* V,
                                 const void* K_hat, const void* V_hat, int n_tok, void* stream);

/* Ragged append (serving batches whose sequences have different lengths; the pages'
 * implementation paragraph describes the write side per token and head, which this applies
 * to each sequence at its own position).  n_tok: host [batch], entries >= 0 (0 leaves a
 * sequence as it is).  K, V (and, for black-box caches, K_hat, V_hat; NULL otherwise) are
 * device arrays of the appended tokens packed sequence by sequence: [sum n_tok][n_kv_heads]
 * [128] of kv_dtype, sequence 0's tokens first.  Sequence i's tokens take positions
 * len_i .. len_i + n_tok[i] - 1.  Once lengths differ the cache keeps per-sequence lengths on
 * the device and every decode attends each sequence over its own length (Tier B's S is that
 * length).  EINVAL if a sequence would exceed max_tokens, ENOMEM if a paged cache's pool has
 * no page left for a new block (nothing is written either way). */
witcert_status witcert_write_ragged(witcert_cache* cache, int layer, const void* K, const void* V,
                                    const void* K_hat, const void* V_hat, const int32_t* n_tok,
                                    void* stream);

/* Empty sequence `seq` in every layer so the slot can serve a new request (continuous
 * batching).  Its repairs are dropped too (their slots in the exact-key pool are not
 * reused), a paged cache returns its pages to the pool, and its value witnesses are zeroed
 * (the decode weighs the rows past a length by 0, which needs finite values there).
 * Asynchronous on `stream`; decodes issued after it see the sequence empty.  EINVAL if
 * seq is out of range. */
witcert_status witcert_reset_sequence(witcert_cache* cache, int seq, void* stream);

/* Fused metered split-KV decode [summary, implementation paragraph (output
 * and meter produced by one kernel reading the cache once, with the
 * certificate terms merged across KV splits by log-sum-exp); Theorem 2
 * (Tier A); Tier B paragraph; improvements list (TV aggregation)].
 * q: device [batch][n_q_heads][128] of kv_dtype, post-RoPE.  Query head j
 * reads KV head j / (Hq/Hkv).  Each sequence attends to all its tokens of `layer`.
 * Outputs (device, caller-owned, float32):
 *   out     [batch][n_q_heads][128]  attention output
 *   meter_a [batch][n_q_heads]       min(1, (A^2-1)/2), A = sum_t p~_t exp(eps_t),
 *                                    eps_t = (1/sqrt d) sum_b ||q_b|| w_{t,b}
 *   meter_b [batch][n_q_heads]       same with c_t = u_t = sqrt(2 s2_t log(2S/delta_loc)),
 *                                    s2_t = (1/d) sum_c q_c^2 s_{c,t}^2/12,
 *                                    delta_loc = delta_req/(L*Hq*T); NaN unless INT8_DITHER
 *   raw_a, raw_b                      the unclamped (A^2-1)/2 of each tier
 *   meter_v [batch][n_q_heads]       value meter E_V = sum_t p~_t wv_t (v_witness caches;
 *                                    EINVAL if non-NULL on a cache without value witnesses)
 * Meters are upper bounds of the formula's value on the stored cache: the sums over
 * tokens, splits and warps are compensated (hi/lo pairs, two-sums), rescaled only by exact powers
 * of two and rounded down (Z) or up (S) where they leave their compensated pairs, and the
 * quotient, D + D^2/2 and a margin of 2^-15 on D are rounded up, so no error grows with the
 * context length; the margin covers each token's own rounding (SFU exponentials and
 * roots, tensor-core products, the expm1 series, which is itself an upper bound) for
 * per-token bounds c_t up to 5 and logits accurate to a few 1e-6.  KIVI2 caches of keys
 * with large outlier channels reach c_t near 30 and logits of tens of units, where the
 * tensor cores' fp32 accumulation of eps_t and of the logits is covered by the margin as
 * measured, not by a worst-case bound.
 * Any meter pointer may be NULL; if all five are NULL the meter work is
 * compiled out and `out` is bit-identical to the metered run's.
 * With the gate enabled, per-16-token-block risks of the gate's tier
 * (Tier B for INT8_DITHER, Tier A otherwise) are kept for witcert_gate.
 * Waits (on the device) for a pending gate of this layer.  An empty layer
 * (len 0) yields zero output and zero meters.  EINVAL on bad arguments. */
witcert_status witcert_decode(witcert_cache* cache, int layer, const void* q, double delta_req,
                              float* out, float* meter_a, float* meter_b, float* raw_a,
                              float* raw_b, float* meter_v, void* stream);

/* Metered decode that allocates nothing.  The paper has no counterpart; this
 * entry point exists for callers that cannot call cudaMalloc while they serve:
 * engines that hand all free device memory to their own pool or caching
 * allocator at start-up (a raw cudaMalloc would then fail, or would bypass that
 * allocator's accounting), and hosts that forbid device allocation outside
 * start-up.  Arguments, results and ordering are those of witcert_decode.  The
 * split-KV partial results live in one static device array of 16 MiB that
 * every GPU loading the library keeps until the process exits; the call rejects
 * with EINVAL a shape whose batch x n_q_heads x KV splits x 544 bytes exceeds
 * it.  The array's device address is looked up (cudaGetSymbolAddress) on the
 * first call made on each device, with that device current; make that first
 * call before any stream capture.  All calls share the array and each call
 * overwrites what it uses (nothing needs to start at zero): calls whose work
 * overlaps on the GPU, on any stream or cache, race and must be serialized by
 * the caller.  No cudaMalloc, cudaFree or allocating library routine is used. */
witcert_status witcert_decode_noalloc(witcert_cache* cache, int layer, const void* q, double delta_req,
                                      float* out, float* meter_a, float* meter_b, float* raw_a,
                                      float* raw_b, float* meter_v, void* stream);

/* Meter-driven gate [summary, implementation paragraph (exact blocks come
 * back from host memory once the meter passes a threshold); Lean page,
 * Figure 2 (repair works on whole blocks and clears their witnesses) and
 * Figure 5 (repairs accumulate and persist)].  Uses the block
 * risks of the layer's last decode: a (sequence, query head) cell whose
 * unrepaired blocks' risks sum to more than D* = sqrt(1+2 tau)-1 (its unclamped
 * meter exceeds tau) has those blocks ranked by risk (largest first, ties to the
 * lower block; a NaN risk counts as +inf) and takes the shortest prefix that leaves
 * remaining risk <= D*.  Sums and comparisons are exact: the fp32 risks are added as
 * integers in units of 2^-149 and compared with D* (float64), so decisions depend on no
 * summation order.  The union over a KV head's query heads is paged in from the pinned
 * backing store into the exact-key pool, marked repaired (persistently) and its witnesses
 * zeroed.  Runs on the cache's side stream after the work already queued on `stream`; later
 * writes and decodes of this layer wait for it on the device.  Repairs affect decodes
 * issued after this call.  ESTATE if the gate is disabled or the layer has not been decoded
 * since its last write.  EPAGEIN, with nothing selected, paged in or zeroed, if the layer's
 * backing store has lost exact keys (a host copy into it failed, or a fault was injected
 * with witcert_inject_fault): its witnesses stay and keep bounding the error. */
witcert_status witcert_gate(witcert_cache* cache, int layer, float tau, void* stream);

/* Gate counters, summed over all gate calls.  Waits for outstanding gate work
 * with a host deadline of `timeout_ms` (ETIMEDOUT if it runs out). */
witcert_status witcert_gate_stats(witcert_cache* cache, witcert_gate_counters* out, int timeout_ms);

/* Context-parallel decode, one shard: this cache holds one slice of a longer context (its
 * tokens at global positions pos_offset, pos_offset + 1, ...; see witcert_config).  The
 * shard's decode of `layer` is merged over the shard's own splits but not normalized: for
 * every (sequence, query head) cell it writes one record of 136 floats to `part` (device,
 * [batch][n_q_heads][136]): m, an integer (log2 units) at least the largest logit (-inf
 * for an empty slice), Z = sum 2^(l - m) rounded down, S_A and S_B = sum 2^(l - m) expm1(c)
 * of the Tier A and Tier B bounds rounded up, S_V = sum 2^(l - m) wv rounded up (0 without
 * value witnesses), three unused floats, and the 128 value sums relative to m.  Tier B's kappa uses s_total, the whole context's
 * length (>= this slice's), so the shards of one decode share delta_loc.  The records of all
 * shards, gathered in any order into [batch][n_q_heads][n_parts][136], are merged by
 * witcert_merge_partials into the same output and meters a single cache holding the whole
 * context would give (up to floating-point summation order).  Block risks are not kept
 * (gating needs a whole-context decode).  Same-stream ordering as witcert_decode. */
witcert_status witcert_decode_partial(witcert_cache* cache, int layer, const void* q, double delta_req,
                                      long long s_total, float* part, void* stream);

/* Merge of context-parallel shard records (see witcert_decode_partial; the log-sum-exp merge
 * of the pages' split-KV decode, applied across shards): parts is device [batch][n_q_heads]
 * [n_parts][136]; out [batch][n_q_heads][128] fp32 and the optional meters [batch][n_q_heads]
 * as in witcert_decode (meter_b NaN unless scheme is WITCERT_INT8_DITHER; meter_v from the
 * records' S_V).  Every record's m must be an integer or -inf, as witcert_decode_partial
 * writes it.  Asynchronous on `stream`; no cache is involved. */
witcert_status witcert_merge_partials(const float* parts, int n_parts, int batch, int n_q_heads,
                                      witcert_scheme scheme, float* out, float* meter_a, float* meter_b,
                                      float* raw_a, float* raw_b, float* meter_v, void* stream);

/* The gate's block selection on its own [summary, implementation paragraph; Lean page,
 * Figure 2], for risks computed elsewhere (the shards of a context-parallel decode combine
 * theirs) and for tests: the rule of witcert_gate, applied to caller arrays.
 *   risk      device float [batch][n_q_heads][nblk]  block risks of each cell
 *   repaired  device uint8 [batch][n_kv_heads][nblk] nonzero = already repaired (not ranked),
 *             or NULL (none repaired)
 *   selected  device uint32 [batch][n_kv_heads][nblk/32 + 1] output bitmap: bit b % 32 of word
 *             b / 32 is set when any query head of the KV head's group selects block b;
 *             cleared by the call first
 * Asynchronous on `stream`.  EINVAL for nblk outside [1, 16384] or bad shapes. */
witcert_status witcert_gate_select(const float* risk, const uint8_t* repaired, int batch, int n_q_heads,
                                   int n_kv_heads, int nblk, float tau, uint32_t* selected, void* stream);

typedef enum {
  WITCERT_FAULT_BACKING_LOST = 1   /* the layer's pinned backing store loses its exact keys, as
                                      when a host copy into it fails */
} witcert_fault;

/* Host-side fault injection for failure-detection tests (no counterpart in the paper): puts
 * `layer` of the cache into the state `fault` describes, as the failure itself would.  With
 * WITCERT_FAULT_BACKING_LOST the layer's gate calls return WITCERT_EPAGEIN from then on and
 * change nothing; decodes are unaffected.  No GPU work.  EINVAL for a bad layer or fault,
 * ESTATE if the gate is disabled. */
witcert_status witcert_inject_fault(witcert_cache* cache, witcert_fault fault, int layer);

/* Library counters.  Synchronizes the device. */
witcert_status witcert_stats(witcert_cache* cache, witcert_stats_t* out);

/* Turn per-launch CUDA-event timing of the decode split kernel on (1) or off (0). */
witcert_status witcert_set_profiling(witcert_cache* cache, int on);

/* Launch overlap (1, the default) or strict serialization (0) of the cache's
 * kernels on a stream.  With overlap, write, decode and merge kernels are
 * launched as programmatic dependents: each may start before its predecessor
 * finishes and waits for it only where it reads or overwrites that
 * predecessor's results.  Results are identical either way. */
witcert_status witcert_set_launch_overlap(witcert_cache* cache, int on);

/* Length of `layer`'s longest sequence (host, synchronous, no device work). */
witcert_status witcert_length(const witcert_cache* cache, int layer, int* len);

/* Length of sequence `seq` in `layer` (host, synchronous, no device work). */
witcert_status witcert_seq_length(const witcert_cache* cache, int layer, int seq, int* len);

/* What witcert_export copies out (layouts below). */
typedef enum {
  WITCERT_X_K_CODES = 0, WITCERT_X_V_CODES = 1, WITCERT_X_K_SCALES = 2, WITCERT_X_V_SCALES = 3,
  WITCERT_X_V_ZEROS = 4, WITCERT_X_KIVI_K_SCALE = 5, WITCERT_X_KIVI_K_ZERO = 6,
  WITCERT_X_WITNESS = 7, WITCERT_X_SLOTS = 8, WITCERT_X_BLOCK_RISK = 9, WITCERT_X_V_WITNESS = 10
} witcert_export_kind;

/* Cache contents in a canonical layout, for inspection and tests.  Writes
 * into a caller-owned device buffer of `bytes` bytes (EINVAL if too small):
 *   WITCERT_X_K_CODES, V_CODES  uint8 [batch][len][n_kv_heads][128]
 *                               (INT8: two's-complement int8; FP8: E4M3 bits;
 *                               KIVI: 0..3, keys of an unfinished block 0);
 *                               BLACKBOX: the stored bf16 values [batch][len][n_kv_heads][128]
 *   WITCERT_X_K_SCALES, V_SCALES fp16 [batch][len][n_kv_heads][4] (INT8; KIVI V scales)
 *   WITCERT_X_V_ZEROS           fp16 [batch][len][n_kv_heads][4] (KIVI)
 *   WITCERT_X_KIVI_K_SCALE, _ZERO fp16 [batch][nblk][n_kv_heads][128] (KIVI, full blocks)
 *   WITCERT_X_WITNESS           fp16 [batch][len][n_kv_heads][16]
 *   WITCERT_X_SLOTS             int32 [batch][n_kv_heads][nblk] (-1 = not repaired)
 *   WITCERT_X_BLOCK_RISK        float [batch][n_q_heads][nblk] (last decode; gate enabled)
 *   WITCERT_X_V_WITNESS         fp16 [batch][len][n_kv_heads] (v_witness caches)
 * nblk = ceil(len/16).  Asynchronous on `stream`. */
witcert_status witcert_export(witcert_cache* cache, int layer, witcert_export_kind what,
                              void* dst, size_t bytes, void* stream);

/* The dither stream xi the INT8 writer and decoder regenerate [summary, Tier B
 * paragraph: the decoder recomputes the same dither instead of storing it], for tests:
 * Philox4x32-10 (Salmon et al., SC'11) with key (seed mod 2^32, seed div 2^32)
 * and counter (t, (c/4) | tensor<<16, kv_head | layer<<16, 0); channel c takes
 * output word c mod 4, xi = (u >> 8) * 2^-24 - 1/2.  Writes float32
 * [n][128] for positions t0..t0+n-1 to device `out`.  tensor 0 = K, 1 = V. */
witcert_status witcert_dither(uint64_t seed, int layer, int kv_head, int t0, int n, int tensor,
                              float* out, void* stream);

/* Failure-detection self test (no counterpart in the paper): runs, on `stream`,
 * the bounded shared-memory barrier wait that the decode pipeline uses, against a
 * barrier that nothing completes, with a limit of `limit_ns` nanoseconds (at most
 * 1e10).  Returns WITCERT_ETIMEDOUT when the wait gives up as designed (the CUDA
 * context stays usable), WITCERT_OK if it was satisfied.  Synchronizes `stream`. */
witcert_status witcert_wait_selftest(int64_t limit_ns, void* stream);

/* Self test of the writers' quotient x / s (no counterpart in the paper): the INT8 writer
 * divides by its fp16 scale s with a reciprocal and one exact correction instead of an IEEE
 * division; this compares the two, on the GPU, for every positive fp16 scale against every
 * bfloat16 x with |x| <= 127.5 s and n_f32 (<= 2^20) seeded float32 x per scale, wherever the
 * quotient can move a code (|x / s| >= 2^-25).  Writes the number of differing quotients to
 * host *mismatches (expected 0).  Synchronizes `stream`. */
witcert_status witcert_quotient_selftest(int n_f32, uint64_t seed, uint64_t* mismatches, void* stream);

/* Thread-local message of the last failing call on this thread ("" if none). */
const char* witcert_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* WITCERT_H */
