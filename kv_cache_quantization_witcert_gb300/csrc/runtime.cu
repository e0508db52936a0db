// Host runtime behind the C ABI in include/witcert.h: owns the cache's device
// pools, the pinned backing store, the side stream of the gate and the events
// that order it against writes and decodes; validates every argument and maps
// failures to status codes with a thread-local message.
#include <chrono>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "../../include/witcert.h"
#include "common.cuh"
#include "kernels.h"

using namespace witcert;

namespace {

thread_local std::string g_err;

witcert_status fail(witcert_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}
witcert_status cuda_fail(cudaError_t e, const char* where) {
  return fail(e == cudaErrorMemoryAllocation ? WITCERT_ENOMEM : WITCERT_ECUDA, "%s: %s", where, cudaGetErrorString(e));
}
void ok() { g_err.clear(); }

struct ProfPair { cudaEvent_t a, b; };

}  // namespace

struct witcert_cache {
  witcert_config cfg{};
  int device = 0, sm_count = 0, scheme = 0, bblk = 0, nblk_max = 0, elem = 0, max_splits = 1;
  size_t layer_blocks = 0;          // bytes of one layer's block store
  uint8_t* blocks = nullptr;
  float* kivi_tail = nullptr;       // [L][B][Hkv][16][128]
  __half* vwit = nullptr;           // [L][B][Hkv][nblk_max][16] value witnesses (v_witness caches)
  int32_t* slots = nullptr;         // [L][B][Hkv][nblk_max]
  void* pool = nullptr;             // [cap][16][128] kv dtype
  void* backing_host = nullptr;     // [L][B][Hkv][max_tokens][128] kv dtype, pinned + mapped
  void* backing_dev = nullptr;
  float2* risk_raw = nullptr;       // [B][Hq][nblk_max]
  float* risk = nullptr;            // [L][B][Hq][nblk_max]
  float* part = nullptr;            // [B][Hq][max_splits][kPartStride]
  uint32_t* selmask = nullptr;
  int4* todo = nullptr;
  unsigned int* todo_count = nullptr;
  unsigned int* pool_next = nullptr;
  unsigned long long* gstats = nullptr;   // [6]
  unsigned long long* clamps = nullptr;
  int* err = nullptr;
  int* dlen = nullptr;              // [L][B] per-sequence lengths on the device (ragged batches)
  int32_t* table = nullptr;         // paged store: [B][nblk_max] page of each block (all layers), -1 = none
  std::vector<int32_t> table_host;  // host copy of the page table
  std::vector<int32_t> free_pages;  // paged store: pages no sequence holds
  std::vector<int> len;             // per layer: the longest sequence
  std::vector<std::vector<int>> slen;   // per layer and sequence
  std::vector<uint64_t> write_gen, risk_gen;   // per layer: writes / resets so far; at the last metered decode
  bool ragged = false;              // sequence lengths may differ: kernels read dlen
  bool lengths_last = false;        // the most recent launch on the cache's stream set dlen
  std::vector<cudaEvent_t> gate_done;
  std::vector<char> gate_pending;
  std::vector<char> backing_lost;   // per layer: the backing store misses exact keys (gate -> EPAGEIN)
  cudaStream_t side = nullptr;
  bool profiling = false;
  std::vector<ProfPair> prof_pending, prof_free;
  double prof_ms = 0.0;
  uint64_t prof_n = 0, tokens_written = 0, decode_calls = 0, gate_calls = 0;
  int last_n_splits = 0;
  bool overlap = true;       // programmatic dependent launch between the cache's kernels
  // most recent launch on the cache's stream when it was a write: its layer and first block
  int last_write_layer = -1, last_write_blk = 0;
};

namespace {

// Writes of at least this many tokens copy their exact keys to the backing store with the
// copy engines rather than with the write kernels' stores.
constexpr int kBulkBackingTokens = 64;

size_t layer_rows(const witcert_cache* c) { return (size_t)c->cfg.batch * c->cfg.n_kv_heads; }
// Backing-store rows per (sequence, KV head): capacity rounded up to whole 16-token blocks,
// so page-in can always copy a full block.
size_t backing_rows(const witcert_cache* c) { return (size_t)c->nblk_max * kBlk; }
// Value witnesses of one layer: [B][Hkv][nblk_max][16].
size_t vwit_layer(const witcert_cache* c) { return layer_rows(c) * c->nblk_max * kBlk; }

witcert_status check_layer(const witcert_cache* c, int layer) {
  if (!c) return fail(WITCERT_EINVAL, "cache is NULL");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(WITCERT_EINVAL, "layer %d out of range [0, %d)", layer, c->cfg.n_layers);
  return WITCERT_OK;
}

void free_all(witcert_cache* c) {
  cudaFree(c->blocks); cudaFree(c->kivi_tail); cudaFree(c->vwit); cudaFree(c->slots); cudaFree(c->pool);
  if (c->backing_host) cudaFreeHost(c->backing_host);
  cudaFree(c->risk_raw); cudaFree(c->risk); cudaFree(c->part); cudaFree(c->selmask); cudaFree(c->todo);
  cudaFree(c->todo_count); cudaFree(c->pool_next); cudaFree(c->gstats); cudaFree(c->clamps); cudaFree(c->err);
  cudaFree(c->dlen); cudaFree(c->table);
  for (auto e : c->gate_done) if (e) cudaEventDestroy(e);
  for (auto& p : c->prof_pending) { cudaEventDestroy(p.a); cudaEventDestroy(p.b); }
  for (auto& p : c->prof_free) { cudaEventDestroy(p.a); cudaEventDestroy(p.b); }
  if (c->side) cudaStreamDestroy(c->side);
}

template <typename T>
cudaError_t dalloc(T** p, size_t bytes) {
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), bytes ? bytes : 16);
  if (e == cudaSuccess) e = cudaMemset(*p, 0, bytes ? bytes : 16);
  return e;
}

// Wait for the gate of `layer` (device-side) before touching that layer again.
// Returns true when it inserted an event wait (the next launch then goes without PDL).
bool order_after_gate(witcert_cache* c, int layer, cudaStream_t st) {
  if (!c->gate_pending[layer]) return false;
  cudaStreamWaitEvent(st, c->gate_done[layer], 0);
  return true;
}

void collect_profile(witcert_cache* c) {
  for (auto& p : c->prof_pending) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) { c->prof_ms += ms; ++c->prof_n; }
    c->prof_free.push_back(p);
  }
  c->prof_pending.clear();
}

}  // namespace

extern "C" {

const char* witcert_last_error(void) { return g_err.c_str(); }

static int auto_splits(const witcert_cache* c, int nblk, bool meter, int cap);

witcert_status witcert_create(const witcert_config* cfg, witcert_cache** out) {
  if (!cfg || !out) return fail(WITCERT_EINVAL, "NULL argument");
  *out = nullptr;
  const witcert_config& f = *cfg;
  if (f.head_dim != 128) return fail(WITCERT_EINVAL, "head_dim must be 128 (got %d)", f.head_dim);
  if (f.n_layers <= 0 || f.n_layers > 65535) return fail(WITCERT_EINVAL, "n_layers must be in [1, 65535]");
  if (f.n_kv_heads <= 0 || f.n_kv_heads > 65535 || f.n_q_heads <= 0 || f.n_q_heads % f.n_kv_heads)
    return fail(WITCERT_EINVAL, "n_q_heads must be a positive multiple of n_kv_heads");
  if (f.n_q_heads / f.n_kv_heads > kMaxGroupHeads) return fail(WITCERT_EINVAL, "at most %d query heads per KV head", kMaxGroupHeads);
  if (f.batch <= 0 || f.max_tokens <= 0) return fail(WITCERT_EINVAL, "batch and max_tokens must be positive");
  if (f.scheme < WITCERT_INT8_DITHER || f.scheme > WITCERT_BLACKBOX) return fail(WITCERT_EINVAL, "unknown scheme %d", (int)f.scheme);
  if (f.kv_dtype != WITCERT_F32 && f.kv_dtype != WITCERT_BF16) return fail(WITCERT_EINVAL, "unknown dtype %d", (int)f.kv_dtype);
  if (f.total_steps <= 0) return fail(WITCERT_EINVAL, "total_steps must be positive");
  if (f.n_splits < 0 || f.max_repair_blocks < 0) return fail(WITCERT_EINVAL, "n_splits and max_repair_blocks must be >= 0");
  if (f.pos_offset < 0) return fail(WITCERT_EINVAL, "pos_offset must be >= 0");
  if (f.max_pages < 0) return fail(WITCERT_EINVAL, "max_pages must be >= 0");
  if (f.max_pages > 0 && f.kv_dtype != WITCERT_BF16) return fail(WITCERT_EINVAL, "a paged cache holds bf16 keys and values");
  if (f.max_repair_blocks > 0 && (f.max_tokens + kBlk - 1) / kBlk > gate_max_blocks())
    return fail(WITCERT_EINVAL, "with the gate enabled max_tokens must be at most %d (the gate ranks up to %d blocks)",
                gate_max_blocks() * kBlk, gate_max_blocks());

  auto* c = new (std::nothrow) witcert_cache();
  if (!c) return fail(WITCERT_ENOMEM, "host allocation failed");
  c->cfg = f;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device);
  if (e != cudaSuccess) { delete c; return cuda_fail(e, "device query"); }
  c->scheme = (int)f.scheme;
  c->bblk = block_bytes(c->scheme);
  c->nblk_max = (f.max_tokens + kBlk - 1) / kBlk;
  c->elem = f.kv_dtype == WITCERT_BF16 ? 2 : 4;
  c->layer_blocks = f.max_pages > 0 ? (size_t)f.max_pages * f.n_kv_heads * c->bblk : layer_rows(c) * c->nblk_max * c->bblk;
  const int auto_on = auto_splits(c, c->nblk_max, true, 0), auto_off = auto_splits(c, c->nblk_max, false, 0);
  const int auto_max = auto_on > auto_off ? auto_on : auto_off;
  c->max_splits = f.n_splits > auto_max ? f.n_splits : auto_max;
  c->len.assign(f.n_layers, 0);
  c->slen.assign(f.n_layers, std::vector<int>(f.batch, 0));
  c->write_gen.assign(f.n_layers, 0);
  c->risk_gen.assign(f.n_layers, ~uint64_t(0));
  c->gate_done.assign(f.n_layers, nullptr);
  c->gate_pending.assign(f.n_layers, 0);
  c->backing_lost.assign(f.n_layers, 0);
  const size_t L = f.n_layers, cells = (size_t)f.batch * f.n_q_heads;
  const bool gate = f.max_repair_blocks > 0;

#define TRY(x, what) do { e = (x); if (e != cudaSuccess) { free_all(c); delete c; return cuda_fail(e, what); } } while (0)
  TRY(dalloc(&c->blocks, L * c->layer_blocks), "allocating the block store");
  if (c->scheme == kKivi) TRY(dalloc(&c->kivi_tail, L * layer_rows(c) * kBlk * kD * sizeof(float)), "allocating the KIVI tail");
  if (f.v_witness) TRY(dalloc(&c->vwit, L * vwit_layer(c) * sizeof(__half)), "allocating value witnesses");
  TRY(dalloc(&c->part, cells * c->max_splits * kPartStride * sizeof(float)), "allocating split scratch");
  TRY(dalloc(&c->clamps, sizeof(unsigned long long)), "allocating counters");
  TRY(dalloc(&c->err, sizeof(int)), "allocating the error word");
  TRY(dalloc(&c->dlen, L * f.batch * sizeof(int)), "allocating sequence lengths");
  if (f.max_pages > 0) {
    const size_t entries = (size_t)f.batch * c->nblk_max;
    TRY(dalloc(&c->table, entries * sizeof(int32_t)), "allocating the page table");
    TRY(cudaMemset(c->table, 0xFF, entries * sizeof(int32_t)), "clearing the page table");
    c->table_host.assign(entries, -1);
    for (int pg = f.max_pages - 1; pg >= 0; --pg) c->free_pages.push_back(pg);
  }
  if (gate) {
    TRY(dalloc(&c->slots, L * layer_rows(c) * c->nblk_max * sizeof(int32_t)), "allocating repair slots");
    TRY(cudaMemset(c->slots, 0xFF, L * layer_rows(c) * c->nblk_max * sizeof(int32_t)), "clearing repair slots");
    TRY(dalloc(&c->pool, (size_t)f.max_repair_blocks * kBlk * kD * c->elem), "allocating the exact-key pool");
    const size_t bbytes = L * layer_rows(c) * (size_t)c->nblk_max * kBlk * kD * c->elem;
    TRY(cudaHostAlloc(&c->backing_host, bbytes, cudaHostAllocMapped), "allocating the pinned backing store");
    memset(c->backing_host, 0, bbytes);
    TRY(cudaHostGetDevicePointer(&c->backing_dev, c->backing_host, 0), "mapping the backing store");
    TRY(dalloc(&c->risk_raw, cells * c->nblk_max * sizeof(float2)), "allocating block-risk scratch");
    TRY(dalloc(&c->risk, L * cells * c->nblk_max * sizeof(float)), "allocating block risks");
    TRY(dalloc(&c->selmask, layer_rows(c) * (c->nblk_max / 32 + 1) * sizeof(uint32_t)), "allocating gate masks");
    TRY(dalloc(&c->todo, layer_rows(c) * c->nblk_max * sizeof(int4)), "allocating the gate todo list");
    TRY(dalloc(&c->todo_count, sizeof(unsigned int)), "allocating gate counters");
    TRY(dalloc(&c->pool_next, sizeof(unsigned int)), "allocating gate counters");
    TRY(dalloc(&c->gstats, 6 * sizeof(unsigned long long)), "allocating gate counters");
    TRY(cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking), "creating the gate stream");
    for (auto& ev : c->gate_done) TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming), "creating gate events");
  }
#undef TRY
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) { free_all(c); delete c; return cuda_fail(e, "create"); }
  *out = c;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_destroy(witcert_cache* c) {
  if (!c) return fail(WITCERT_EINVAL, "cache is NULL");
  cudaDeviceSynchronize();
  free_all(c);
  delete c;
  ok();
  return WITCERT_OK;
}

// Write arguments of `layer` for all sequences: appends of n_tok tokens at t0.
static WriteArgs layer_write_args(const witcert_cache* c, int layer, const void* K, const void* V, const void* Kh,
                                  const void* Vh, int n_tok, int t0) {
  WriteArgs a{};
  a.blocks = c->blocks + layer * c->layer_blocks;
  a.table = c->table;
  a.nblk_max = c->nblk_max;
  a.K = K; a.V = V; a.Kh = Kh; a.Vh = Vh;
  if (c->vwit) a.vwit = c->vwit + layer * vwit_layer(c);
  a.B = c->cfg.batch; a.Hkv = c->cfg.n_kv_heads; a.n_tok = n_tok; a.t0 = t0; a.layer = layer;
  a.backing_rows = (int)backing_rows(c);
  a.is_bf16 = c->cfg.kv_dtype == WITCERT_BF16;
  a.seed = c->cfg.seed;
  philox_round_keys(a.seed, a.rk0, a.rk1);
  a.pos0 = c->cfg.pos_offset;
  if (c->backing_dev)
    a.backing = static_cast<uint8_t*>(c->backing_dev) + layer * layer_rows(c) * backing_rows(c) * kD * c->elem;
  if (c->slots) a.slots = c->slots + layer * layer_rows(c) * c->nblk_max;
  a.pool = c->pool;
  if (c->kivi_tail) a.kivi_tail = c->kivi_tail + layer * layer_rows(c) * kBlk * kD;
  a.clamps = c->clamps;
  return a;
}

// The same arguments narrowed to sequence i alone (B = 1): its n tokens sit at packed input
// row in_row (tokens, each n_kv_heads x 128 elements) and are appended at position t0.
static WriteArgs seq_write_args(const witcert_cache* c, const WriteArgs& all, int i, size_t in_row, int n, int t0) {
  WriteArgs a = all;
  const size_t rows = (size_t)i * c->cfg.n_kv_heads;          // (sequence, KV head) rows before i
  const size_t in_bytes = in_row * c->cfg.n_kv_heads * kD * c->elem;
  if (a.table) a.table += (size_t)i * c->nblk_max;            // paged: the sequence's row of the table
  else a.blocks += rows * c->nblk_max * c->bblk;
  if (a.vwit) a.vwit += rows * c->nblk_max * kBlk;
  if (a.backing) a.backing = static_cast<uint8_t*>(a.backing) + rows * backing_rows(c) * kD * c->elem;
  if (a.slots) a.slots += rows * c->nblk_max;
  if (a.kivi_tail) a.kivi_tail += rows * kBlk * kD;
  a.K = static_cast<const uint8_t*>(all.K) + in_bytes;
  a.V = static_cast<const uint8_t*>(all.V) + in_bytes;
  if (all.Kh) a.Kh = static_cast<const uint8_t*>(all.Kh) + in_bytes;
  if (all.Vh) a.Vh = static_cast<const uint8_t*>(all.Vh) + in_bytes;
  a.B = 1; a.n_tok = n; a.t0 = t0;
  return a;
}

// Device copies of per-sequence lengths: entries (layer * batch + sequence, length), sent as
// kernel parameters (no host buffer outlives the call).
static cudaError_t push_ints(int* dst, const std::vector<std::pair<int, int>>& upd, cudaStream_t st, bool& pdl) {
  for (size_t k0 = 0; k0 < upd.size(); k0 += kRaggedPerLaunch) {
    LengthArgs u{};
    u.dst = dst;
    for (size_t k = k0; k < upd.size() && k < k0 + kRaggedPerLaunch; ++k) {
      u.idx[u.n] = upd[k].first;
      u.len[u.n] = upd[k].second;
      ++u.n;
    }
    cudaError_t e = launch_set_lengths(u, st, pdl);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
static cudaError_t push_lengths(witcert_cache* c, const std::vector<std::pair<int, int>>& upd, cudaStream_t st,
                                bool& pdl) {
  return push_ints(c->dlen, upd, st, pdl);
}

// Paged store: pages for every block the appends of n touch that has none yet (the table is
// shared by the layers, so the first layer to reach a block takes its page).  Fails, taking
// back what it took, when the pool runs out.
static witcert_status take_pages(witcert_cache* c, int layer, const std::vector<int>& n,
                                 std::vector<std::pair<int, int>>& upd) {
  if (!c->table) return WITCERT_OK;
  for (int i = 0; i < c->cfg.batch; ++i) {
    if (n[i] == 0) continue;
    const int t0 = c->slen[layer][i];
    for (int b = t0 / kBlk; b <= (t0 + n[i] - 1) / kBlk; ++b) {
      int32_t& e = c->table_host[(size_t)i * c->nblk_max + b];
      if (e >= 0) continue;
      if (c->free_pages.empty()) {
        for (auto& u : upd) {
          c->free_pages.push_back(u.second);
          c->table_host[u.first] = -1;
        }
        upd.clear();
        return fail(WITCERT_ENOMEM, "the page pool (%d pages) is exhausted", c->cfg.max_pages);
      }
      e = c->free_pages.back();
      c->free_pages.pop_back();
      upd.emplace_back((int)((size_t)i * c->nblk_max + b), e);
    }
  }
  return WITCERT_OK;
}

// From now on the sequences' lengths may differ: the device gets every layer's lengths.
static cudaError_t enter_ragged(witcert_cache* c, cudaStream_t st, bool& pdl) {
  if (c->ragged) return cudaSuccess;
  std::vector<std::pair<int, int>> upd;
  for (int l = 0; l < c->cfg.n_layers; ++l)
    for (int i = 0; i < c->cfg.batch; ++i) upd.emplace_back(l * c->cfg.batch + i, c->slen[l][i]);
  cudaError_t e = push_lengths(c, upd, st, pdl);
  if (e == cudaSuccess) c->ragged = true;
  return e;
}

// Exact keys of n tokens of sequence i (packed input row in_row) to the pinned backing store
// at position t0, one strided copy-engine transfer per KV head.
static cudaError_t backing_copy(witcert_cache* c, int layer, const void* K, int i, size_t in_row, int n, int t0,
                                cudaStream_t st) {
  const size_t row = (size_t)kD * c->elem;
  const int Hkv = c->cfg.n_kv_heads;
  uint8_t* host = static_cast<uint8_t*>(c->backing_host) + layer * layer_rows(c) * backing_rows(c) * row;
  cudaError_t e = cudaSuccess;
  for (int h = 0; h < Hkv && e == cudaSuccess; ++h)
    e = cudaMemcpy2DAsync(host + (((size_t)i * Hkv + h) * backing_rows(c) + t0) * row, row,
                          static_cast<const uint8_t*>(K) + (in_row * Hkv + h) * row, Hkv * row, row, n,
                          cudaMemcpyDeviceToHost, st);
  return e;
}

// Appends counts[i] tokens (n_uniform each when counts is NULL) to every sequence of `layer`;
// inputs are packed sequence-major.  Equal appends to equal lengths take the batched writers;
// anything else marks the cache ragged and writes each sequence at its own position.
static witcert_status write_impl(witcert_cache* c, int layer, const void* K, const void* V, const void* Kh,
                                 const void* Vh, const int32_t* counts, int n_uniform, void* stream) {
  if (witcert_status s = check_layer(c, layer)) return s;
  const int B = c->cfg.batch;
  std::vector<int> n(B, n_uniform);
  long long total = 0;
  for (int i = 0; i < B; ++i) {
    if (counts) n[i] = counts[i];
    if (n[i] < 0) return fail(WITCERT_EINVAL, "token counts must be >= 0 (sequence %d: %d)", i, n[i]);
    if ((long long)c->slen[layer][i] + n[i] > c->cfg.max_tokens)
      return fail(WITCERT_EINVAL, "layer %d sequence %d would hold %lld tokens, capacity %d", layer, i,
                  (long long)c->slen[layer][i] + n[i], c->cfg.max_tokens);
    total += n[i];
  }
  if (total > 0 && (!K || !V)) return fail(WITCERT_EINVAL, "K and V must not be NULL");
  if (total > 0 && c->scheme == kBbox && (!Kh || !Vh)) return fail(WITCERT_EINVAL, "K_hat and V_hat must not be NULL");
  if (total == 0) { ok(); return WITCERT_OK; }
  bool uniform = !c->ragged;
  for (int i = 1; i < B && uniform; ++i) uniform = n[i] == n[0];
  std::vector<std::pair<int, int>> pages;
  if (witcert_status ps = take_pages(c, layer, n, pages)) return ps;
  auto st = static_cast<cudaStream_t>(stream);
  const bool waited = order_after_gate(c, layer, st);
  bool pdl = c->overlap && !waited;
  cudaError_t e = push_ints(c->table, pages, st, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "page table");
  int first_blk = INT_MAX;
  if (uniform) {
    const int n_tok = n[0], t0 = c->len[layer];
    WriteArgs a = layer_write_args(c, layer, K, V, Kh, Vh, n_tok, t0);
    // a page-table update launched just before must be complete before the writers read it
    a.late_wait = pages.empty();
    if (c->backing_host && n_tok >= kBulkBackingTokens) {
      // bulk writes copy their exact keys to the pinned backing store with the copy engines
      // instead of the kernels' stores over C2C
      for (int i = 0; i < B && e == cudaSuccess; ++i) e = backing_copy(c, layer, K, i, (size_t)i * n_tok, n_tok, t0, st);
      if (e != cudaSuccess) {
        c->backing_lost[layer] = 1;
        return cuda_fail(e, "backing-store copy");
      }
      a.backing = nullptr;
      pdl = false;                     // the copies sit between this write and its predecessor
    }
    e = launch_write(c->scheme, a, st, pdl);
    if (e != cudaSuccess) return cuda_fail(e, "write launch");
    first_blk = t0 / kBlk;
  } else {
    if ((e = enter_ragged(c, st, pdl)) != cudaSuccess) return cuda_fail(e, "sequence lengths");
    std::vector<std::pair<int, int>> upd;
    for (int i = 0; i < B; ++i)
      if (n[i] > 0) upd.emplace_back(layer * B + i, c->slen[layer][i] + n[i]);
    if ((e = push_lengths(c, upd, st, pdl)) != cudaSuccess) return cuda_fail(e, "sequence lengths");
    const WriteArgs all = layer_write_args(c, layer, K, V, Kh, Vh, 0, 0);
    // long appends: the batched writers on that sequence alone; short ones: ragged launches
    // of up to kRaggedPerLaunch sequences
    RaggedArgs g{};
    auto flush = [&]() -> cudaError_t {
      if (g.n_seq == 0) return cudaSuccess;
      cudaError_t r = launch_write_ragged(c->scheme, all, g, st, pdl);
      // KIVI keys close per 16-token block: each sequence's blocks by its own launch
      for (int k = 0; k < g.n_seq && r == cudaSuccess && c->scheme == kKivi; ++k)
        r = launch_kivi_keys(seq_write_args(c, all, g.seq[k], (size_t)g.row0[k], g.off[k + 1] - g.off[k], g.t0[k]),
                             st, pdl);
      g = RaggedArgs{};
      return r;
    };
    size_t row = 0;
    for (int i = 0; i < B && e == cudaSuccess; ++i) {
      if (n[i] == 0) continue;
      const int t0 = c->slen[layer][i];
      first_blk = t0 / kBlk < first_blk ? t0 / kBlk : first_blk;
      if (n[i] >= kBlk) {
        WriteArgs a = seq_write_args(c, all, i, row, n[i], t0);
        if (c->backing_host && n[i] >= kBulkBackingTokens) {
          e = backing_copy(c, layer, K, i, row, n[i], t0, st);
          if (e != cudaSuccess) {
            c->backing_lost[layer] = 1;
            return cuda_fail(e, "backing-store copy");
          }
          a.backing = nullptr;
          pdl = false;
        }
        e = launch_write(c->scheme, a, st, pdl);
      } else {
        g.seq[g.n_seq] = i;
        g.t0[g.n_seq] = t0;
        g.row0[g.n_seq] = (int)row;
        g.off[g.n_seq + 1] = g.off[g.n_seq] + n[i];
        if (++g.n_seq == kRaggedPerLaunch) e = flush();
      }
      row += n[i];
    }
    if (e == cudaSuccess) e = flush();
    if (e != cudaSuccess) return cuda_fail(e, "ragged write launch");
  }
  c->last_write_layer = layer;
  c->last_write_blk = first_blk;
  c->lengths_last = false;
  for (int i = 0; i < B; ++i) c->slen[layer][i] += n[i];
  int mx = 0;
  for (int i = 0; i < B; ++i) mx = c->slen[layer][i] > mx ? c->slen[layer][i] : mx;
  c->len[layer] = mx;
  ++c->write_gen[layer];
  c->tokens_written += (uint64_t)total * c->cfg.n_kv_heads;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_write(witcert_cache* c, int layer, const void* K, const void* V, int n_tok, void* stream) {
  if (c && c->scheme == kBbox) return fail(WITCERT_EINVAL, "a black-box cache is written with witcert_write_hat");
  if (n_tok < 0) return fail(WITCERT_EINVAL, "n_tok must be >= 0");
  return write_impl(c, layer, K, V, nullptr, nullptr, nullptr, n_tok, stream);
}

witcert_status witcert_write_hat(witcert_cache* c, int layer, const void* K, const void* V, const void* K_hat,
                                 const void* V_hat, int n_tok, void* stream) {
  if (c && c->scheme != kBbox) return fail(WITCERT_EINVAL, "witcert_write_hat needs a WITCERT_BLACKBOX cache");
  if (n_tok < 0) return fail(WITCERT_EINVAL, "n_tok must be >= 0");
  return write_impl(c, layer, K, V, K_hat, V_hat, nullptr, n_tok, stream);
}

witcert_status witcert_write_ragged(witcert_cache* c, int layer, const void* K, const void* V, const void* K_hat,
                                    const void* V_hat, const int32_t* n_tok, void* stream) {
  if (!c || !n_tok) return fail(WITCERT_EINVAL, "cache and n_tok must not be NULL");
  if (c->scheme != kBbox && (K_hat || V_hat)) return fail(WITCERT_EINVAL, "K_hat and V_hat belong to black-box caches");
  return write_impl(c, layer, K, V, K_hat, V_hat, n_tok, 0, stream);
}

witcert_status witcert_reset_sequence(witcert_cache* c, int seq, void* stream) {
  if (!c) return fail(WITCERT_EINVAL, "cache is NULL");
  if (seq < 0 || seq >= c->cfg.batch) return fail(WITCERT_EINVAL, "sequence %d out of range [0, %d)", seq, c->cfg.batch);
  auto st = static_cast<cudaStream_t>(stream);
  bool waited = false;
  for (int l = 0; l < c->cfg.n_layers; ++l) waited |= order_after_gate(c, l, st);
  bool pdl = c->overlap && !waited;
  cudaError_t e = enter_ragged(c, st, pdl);
  std::vector<std::pair<int, int>> upd;
  for (int l = 0; l < c->cfg.n_layers; ++l) upd.emplace_back(l * c->cfg.batch + seq, 0);
  if (e == cudaSuccess) e = push_lengths(c, upd, st, pdl);
  if (c->table && e == cudaSuccess) {       // its pages go back to the pool
    std::vector<std::pair<int, int>> freed;
    for (int b = 0; b < c->nblk_max; ++b) {
      int32_t& pg = c->table_host[(size_t)seq * c->nblk_max + b];
      if (pg < 0) continue;
      c->free_pages.push_back(pg);
      pg = -1;
      freed.emplace_back((int)((size_t)seq * c->nblk_max + b), -1);
    }
    e = push_ints(c->table, freed, st, pdl);
  }
  // the sequence's repairs go with it (their pool slots are not reused)
  const size_t rows = (size_t)c->cfg.n_kv_heads * c->nblk_max;
  for (int l = 0; l < c->cfg.n_layers && e == cudaSuccess && c->slots; ++l)
    e = cudaMemsetAsync(c->slots + (size_t)l * layer_rows(c) * c->nblk_max + (size_t)seq * rows, 0xFF,
                        rows * sizeof(int32_t), st);
  // value witnesses past the next occupant's length are read (with weight 0): keep them zero
  for (int l = 0; l < c->cfg.n_layers && e == cudaSuccess && c->vwit; ++l)
    e = cudaMemsetAsync(c->vwit + l * vwit_layer(c) + (size_t)seq * rows * kBlk, 0, rows * kBlk * sizeof(__half), st);
  if (e != cudaSuccess) return cuda_fail(e, "reset");
  for (int l = 0; l < c->cfg.n_layers; ++l) {
    c->slen[l][seq] = 0;
    int mx = 0;
    for (int i = 0; i < c->cfg.batch; ++i) mx = c->slen[l][i] > mx ? c->slen[l][i] : mx;
    c->len[l] = mx;
    ++c->write_gen[l];
  }
  c->last_write_layer = -1;
  c->lengths_last = true;
  ok();
  return WITCERT_OK;
}

// Automatic split count for a decode of nblk blocks: sized by how many split-kernel CTAs of
// this configuration fit on an SM, and never above the scratch sized at create time.
static int auto_splits(const witcert_cache* c, int nblk, bool meter, int cap) {
  DecodeArgs a{};
  a.B = c->cfg.batch;
  a.is_bf16 = c->cfg.kv_dtype == WITCERT_BF16;
  a.meter = meter;
  a.slots = c->slots;
  const int per_sm = decode_ctas_per_sm(c->scheme, a);
  int s = decode_auto_splits(c->scheme, c->cfg.batch, c->cfg.n_kv_heads, nblk > 0 ? nblk : 1, c->sm_count, per_sm);
  if (cap > 0 && s > cap) s = cap;
  return s;
}

// Decode arguments shared by every decode entry point: the layer's store, the query, the
// split count and the Tier B factor kappa = sqrt(2 ln(2 S / delta_loc)) rounded up, with S
// the attended context (s_kappa; the layer's own length when 0).
static void fill_decode(witcert_cache* c, int layer, const void* q, double delta_req, bool meter, long long s_kappa,
                        DecodeArgs& a) {
  const int S = c->len[layer];
  const int nblk = (S + kBlk - 1) / kBlk;
  a.blocks = c->blocks + layer * c->layer_blocks;
  a.nblk_max = c->nblk_max;
  if (c->slots) a.slots = c->slots + layer * layer_rows(c) * c->nblk_max;
  a.pool = c->pool;
  if (c->kivi_tail) a.kivi_tail = c->kivi_tail + layer * layer_rows(c) * kBlk * kD;
  a.q = q;
  a.is_bf16 = c->cfg.kv_dtype == WITCERT_BF16;
  a.B = c->cfg.batch; a.Hq = c->cfg.n_q_heads; a.Hkv = c->cfg.n_kv_heads; a.grp = a.Hq / a.Hkv; a.S = S;
  if (c->ragged) a.seq_len = c->dlen + (size_t)layer * c->cfg.batch;
  a.table = c->table;
  a.n_splits = c->cfg.n_splits > 0 ? c->cfg.n_splits : auto_splits(c, nblk, meter, c->max_splits);
  a.seed = c->cfg.seed;
  philox_round_keys(a.seed, a.rk0, a.rk1);
  a.layer = layer;
  a.pos0 = c->cfg.pos_offset;
  a.dirty_blk = c->last_write_layer == layer ? c->last_write_blk : INT_MAX;
  float kappa = 0.f;
  const long long Sk = s_kappa > 0 ? s_kappa : S;
  if (meter && Sk > 0) {
    const double dloc = delta_req / ((double)c->cfg.n_layers * c->cfg.n_q_heads * c->cfg.total_steps);
    const double k = std::sqrt(2.0 * std::log(2.0 * (double)Sk / dloc));
    kappa = (float)k;
    if ((double)kappa < k) kappa = std::nextafter(kappa, INFINITY);
  }
  if (meter) a.log2dl = std::log(2.0 * (double)c->cfg.n_layers * c->cfg.n_q_heads * c->cfg.total_steps / delta_req);
  a.kappa = kappa;
  a.err = c->err;
  if (layer + 1 < c->cfg.n_layers && c->len[layer + 1] > 0) a.next_blocks = c->blocks + (layer + 1) * c->layer_blocks;
  if (c->vwit && meter) a.vwit = c->vwit + layer * vwit_layer(c);
  a.meter = meter;
}

witcert_status witcert_decode(witcert_cache* c, int layer, const void* q, double delta_req, float* out,
                              float* meter_a, float* meter_b, float* raw_a, float* raw_b, float* meter_v,
                              void* stream) {
  if (witcert_status s = check_layer(c, layer)) return s;
  if (!q || !out) return fail(WITCERT_EINVAL, "q and out must not be NULL");
  if (meter_v && !c->vwit) return fail(WITCERT_EINVAL, "meter_v needs a cache created with v_witness");
  const bool meter = meter_a || meter_b || raw_a || raw_b || meter_v;
  if (meter && !(delta_req > 0.0 && delta_req <= 1.0)) return fail(WITCERT_EINVAL, "delta_req must be in (0, 1]");
  auto st = static_cast<cudaStream_t>(stream);
  const bool waited = order_after_gate(c, layer, st);
  DecodeArgs a{};
  fill_decode(c, layer, q, delta_req, meter, 0, a);
  a.part = c->part;
  const bool gate = c->cfg.max_repair_blocks > 0;
  if (gate && meter) {
    a.risk_raw = c->risk_raw;
    a.risk = c->risk + (size_t)layer * a.B * a.Hq * c->nblk_max;
  }
  a.out = out; a.meter_a = meter_a; a.meter_b = meter_b; a.raw_a = raw_a; a.raw_b = raw_b; a.meter_v = meter_v;
  ProfPair pp{nullptr, nullptr};
  if (c->profiling) {
    if (c->prof_free.empty()) {
      ProfPair n{};
      if (cudaEventCreate(&n.a) != cudaSuccess || cudaEventCreate(&n.b) != cudaSuccess)
        return fail(WITCERT_ECUDA, "creating profiling events");
      c->prof_free.push_back(n);
    }
    pp = c->prof_free.back();
    c->prof_free.pop_back();
  }
  // the split kernel reads the sequence lengths before it waits for its predecessor
  cudaError_t e = launch_decode(c->scheme, a, c->sm_count, st, pp.a, pp.b, c->overlap && !waited && !c->lengths_last);
  if (pp.a) c->prof_pending.push_back(pp);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  c->lengths_last = false;
  if (gate && meter) c->risk_gen[layer] = c->write_gen[layer];
  c->last_write_layer = -1;
  c->last_n_splits = a.n_splits;
  ++c->decode_calls;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_decode_noalloc(witcert_cache* c, int layer, const void* q, double delta_req, float* out,
                                      float* meter_a, float* meter_b, float* raw_a, float* raw_b, float* meter_v,
                                      void* stream) {
  if (witcert_status s = check_layer(c, layer)) return s;
  if (!q || !out) return fail(WITCERT_EINVAL, "q and out must not be NULL");
  if (meter_v && !c->vwit) return fail(WITCERT_EINVAL, "meter_v needs a cache created with v_witness");
  const bool meter = meter_a || meter_b || raw_a || raw_b || meter_v;
  if (meter && !(delta_req > 0.0 && delta_req <= 1.0)) return fail(WITCERT_EINVAL, "delta_req must be in (0, 1]");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != c->device)
    return fail(WITCERT_EINVAL, "the cache lives on device %d; make it current before this call", c->device);
  DecodeArgs a{};
  fill_decode(c, layer, q, delta_req, meter, 0, a);
  float* scratch = nullptr;
  size_t scratch_bytes = 0;
  cudaError_t e = decode_static_scratch(&scratch, &scratch_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "locating the static split scratch");
  const size_t need = (size_t)a.B * a.Hq * a.n_splits * kPartStride * sizeof(float);
  if (need > scratch_bytes)
    return fail(WITCERT_EINVAL, "batch %d x %d query heads x %d splits needs %zu bytes of split scratch; "
                "the static array holds %zu", a.B, a.Hq, a.n_splits, need, scratch_bytes);
  auto st = static_cast<cudaStream_t>(stream);
  const bool waited = order_after_gate(c, layer, st);
  a.dirty_blk = c->last_write_layer == layer ? c->last_write_blk : INT_MAX;
  a.part = scratch;
  const bool gate = c->cfg.max_repair_blocks > 0;
  if (gate && meter) {
    a.risk_raw = c->risk_raw;
    a.risk = c->risk + (size_t)layer * a.B * a.Hq * c->nblk_max;
  }
  a.out = out; a.meter_a = meter_a; a.meter_b = meter_b; a.raw_a = raw_a; a.raw_b = raw_b; a.meter_v = meter_v;
  e = launch_decode(c->scheme, a, c->sm_count, st, nullptr, nullptr, c->overlap && !waited && !c->lengths_last);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  c->lengths_last = false;
  if (gate && meter) c->risk_gen[layer] = c->write_gen[layer];
  c->last_write_layer = -1;
  c->last_n_splits = a.n_splits;
  ++c->decode_calls;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_decode_partial(witcert_cache* c, int layer, const void* q, double delta_req,
                                      long long s_total, float* part, void* stream) {
  if (witcert_status s = check_layer(c, layer)) return s;
  if (!q || !part) return fail(WITCERT_EINVAL, "q and part must not be NULL");
  if (!(delta_req > 0.0 && delta_req <= 1.0)) return fail(WITCERT_EINVAL, "delta_req must be in (0, 1]");
  if (s_total < c->len[layer]) return fail(WITCERT_EINVAL, "s_total %lld is below the slice's own %d tokens",
                                           s_total, c->len[layer]);
  if (c->ragged) return fail(WITCERT_ESTATE, "context-parallel shards hold equal-length sequences");
  auto st = static_cast<cudaStream_t>(stream);
  const bool waited = order_after_gate(c, layer, st);
  DecodeArgs a{};
  fill_decode(c, layer, q, delta_req, true, s_total, a);
  a.part = c->part;
  a.part_out = part;
  cudaError_t e = launch_decode(c->scheme, a, c->sm_count, st, nullptr, nullptr, c->overlap && !waited);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  c->last_write_layer = -1;
  c->last_n_splits = a.n_splits;
  ++c->decode_calls;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_merge_partials(const float* parts, int n_parts, int batch, int n_q_heads,
                                      witcert_scheme scheme, float* out, float* meter_a, float* meter_b,
                                      float* raw_a, float* raw_b, float* meter_v, void* stream) {
  if (!parts || !out) return fail(WITCERT_EINVAL, "parts and out must not be NULL");
  if (n_parts < 1 || batch < 1 || n_q_heads < 1) return fail(WITCERT_EINVAL, "n_parts, batch and n_q_heads must be >= 1");
  if (scheme < WITCERT_INT8_DITHER || scheme > WITCERT_BLACKBOX) return fail(WITCERT_EINVAL, "unknown scheme %d", (int)scheme);
  DecodeArgs a{};
  a.part = const_cast<float*>(parts);
  a.n_splits = n_parts;
  a.B = batch; a.Hq = n_q_heads;
  a.out = out; a.meter_a = meter_a; a.meter_b = meter_b; a.raw_a = raw_a; a.raw_b = raw_b; a.meter_v = meter_v;
  a.meter = meter_a || meter_b || raw_a || raw_b || meter_v;
  cudaError_t e = launch_merge_records((int)scheme, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  ok();
  return WITCERT_OK;
}

witcert_status witcert_gate(witcert_cache* c, int layer, float tau, void* stream) {
  if (witcert_status s = check_layer(c, layer)) return s;
  if (c->cfg.max_repair_blocks <= 0) return fail(WITCERT_ESTATE, "the gate is disabled (max_repair_blocks = 0)");
  if (!(tau >= 0.f) || !std::isfinite(tau)) return fail(WITCERT_EINVAL, "tau must be finite and >= 0");
  if (c->risk_gen[layer] != c->write_gen[layer] || c->len[layer] == 0)
    return fail(WITCERT_ESTATE, "layer %d has no metered decode since its last write", layer);
  if (c->backing_lost[layer])
    return fail(WITCERT_EPAGEIN, "layer %d: the backing store lost exact keys; nothing was paged in", layer);
  auto st = static_cast<cudaStream_t>(stream);
  cudaEvent_t ready = c->gate_done[layer];
  cudaError_t e = cudaEventRecord(ready, st);   // reuse: marks the point the gate must follow
  if (e == cudaSuccess) e = cudaStreamWaitEvent(c->side, ready, 0);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->todo_count, 0, sizeof(unsigned int), c->side);
  if (e != cudaSuccess) return cuda_fail(e, "gate ordering");
  GateArgs a{};
  const size_t cells = (size_t)c->cfg.batch * c->cfg.n_q_heads;
  a.risk = c->risk + (size_t)layer * cells * c->nblk_max;
  a.slots = c->slots + layer * layer_rows(c) * c->nblk_max;
  a.selmask = c->selmask; a.todo = c->todo; a.todo_count = c->todo_count; a.pool_next = c->pool_next;
  a.stats = c->gstats;
  a.blocks = c->blocks + layer * c->layer_blocks;
  a.backing = static_cast<uint8_t*>(c->backing_dev) + layer * layer_rows(c) * backing_rows(c) * kD * c->elem;
  a.pool = c->pool;
  a.nblk_max = c->nblk_max; a.B = c->cfg.batch; a.Hq = c->cfg.n_q_heads; a.Hkv = c->cfg.n_kv_heads;
  a.grp = a.Hq / a.Hkv; a.S = c->len[layer]; a.backing_rows = (int)backing_rows(c);
  if (c->ragged) a.seq_len = c->dlen + (size_t)layer * c->cfg.batch;
  a.table = c->table;
  a.pool_capacity = c->cfg.max_repair_blocks; a.scheme = c->scheme; a.elem_bytes = c->elem;
  a.d_star = std::sqrt(1.0 + 2.0 * (double)tau) - 1.0;
  e = launch_gate(a, c->side);
  if (e == cudaSuccess) e = cudaEventRecord(c->gate_done[layer], c->side);
  if (e != cudaSuccess) return cuda_fail(e, "gate launch");
  c->gate_pending[layer] = 1;
  ++c->gate_calls;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_gate_select(const float* risk, const uint8_t* repaired, int batch, int n_q_heads,
                                   int n_kv_heads, int nblk, float tau, uint32_t* selected, void* stream) {
  if (!risk || !selected) return fail(WITCERT_EINVAL, "risk and selected must not be NULL");
  if (batch < 1 || n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads)
    return fail(WITCERT_EINVAL, "batch >= 1 and n_q_heads a positive multiple of n_kv_heads");
  if (nblk < 1 || nblk > gate_max_blocks()) return fail(WITCERT_EINVAL, "nblk must be in [1, %d]", gate_max_blocks());
  if (!(tau >= 0.f) || !std::isfinite(tau)) return fail(WITCERT_EINVAL, "tau must be finite and >= 0");
  auto st = static_cast<cudaStream_t>(stream);
  GateArgs a{};
  a.risk = risk;
  a.repaired = repaired;
  a.selmask = selected;
  a.nblk_max = nblk; a.B = batch; a.Hq = n_q_heads; a.Hkv = n_kv_heads; a.grp = n_q_heads / n_kv_heads;
  a.S = nblk * kBlk;
  a.d_star = std::sqrt(1.0 + 2.0 * (double)tau) - 1.0;
  cudaError_t e = cudaMemsetAsync(selected, 0, (size_t)batch * n_kv_heads * (nblk / 32 + 1) * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = launch_gate_select(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "gate selection");
  ok();
  return WITCERT_OK;
}

witcert_status witcert_inject_fault(witcert_cache* c, witcert_fault fault, int layer) {
  if (witcert_status s = check_layer(c, layer)) return s;
  if (fault != WITCERT_FAULT_BACKING_LOST) return fail(WITCERT_EINVAL, "unknown fault %d", (int)fault);
  if (c->cfg.max_repair_blocks <= 0) return fail(WITCERT_ESTATE, "the gate is disabled: there is no backing store");
  c->backing_lost[layer] = 1;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_gate_stats(witcert_cache* c, witcert_gate_counters* out, int timeout_ms) {
  if (!c || !out) return fail(WITCERT_EINVAL, "NULL argument");
  memset(out, 0, sizeof *out);
  out->gate_calls = c->gate_calls;
  if (c->cfg.max_repair_blocks <= 0) { ok(); return WITCERT_OK; }
  const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms < 0 ? 0 : timeout_ms);
  for (int l = 0; l < c->cfg.n_layers; ++l) {
    if (!c->gate_pending[l]) continue;
    for (;;) {
      cudaError_t q = cudaEventQuery(c->gate_done[l]);
      if (q == cudaSuccess) break;
      if (q != cudaErrorNotReady) return cuda_fail(q, "gate event");
      if (std::chrono::steady_clock::now() > deadline) return fail(WITCERT_ETIMEDOUT, "gate of layer %d still running", l);
      std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
  }
  unsigned long long s[6] = {0, 0, 0, 0, 0, 0};
  cudaError_t e = cudaMemcpy(s, c->gstats, sizeof s, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading gate counters");
  out->cells_triggered = s[0]; out->blocks_selected = s[1]; out->blocks_paged_in = s[2];
  out->bytes_paged_in = s[3]; out->blocks_dropped = s[4];
  ok();
  return WITCERT_OK;
}

witcert_status witcert_stats(witcert_cache* c, witcert_stats_t* out) {
  if (!c || !out) return fail(WITCERT_EINVAL, "NULL argument");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "stats");
  memset(out, 0, sizeof *out);
  unsigned long long cl = 0;
  int er = 0;
  if ((e = cudaMemcpy(&cl, c->clamps, sizeof cl, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e, "stats");
  if ((e = cudaMemcpy(&er, c->err, sizeof er, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e, "stats");
  collect_profile(c);
  out->tokens_written = c->tokens_written;
  out->decode_calls = c->decode_calls;
  out->int8_clamps = cl;
  out->device_errors = (uint64_t)er;
  out->decode_kernel_ms = c->prof_ms;
  out->decode_kernel_launches = c->prof_n;
  out->last_n_splits = c->last_n_splits;
  out->pages_used = c->table ? (uint64_t)c->cfg.max_pages - c->free_pages.size() : 0;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_set_profiling(witcert_cache* c, int on) {
  if (!c) return fail(WITCERT_EINVAL, "cache is NULL");
  if (!on && c->profiling) {
    cudaDeviceSynchronize();
    collect_profile(c);
  }
  if (on && !c->profiling) { cudaDeviceSynchronize(); collect_profile(c); c->prof_ms = 0.0; c->prof_n = 0; }
  c->profiling = on != 0;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_set_launch_overlap(witcert_cache* c, int on) {
  if (!c) return fail(WITCERT_EINVAL, "cache is NULL");
  c->overlap = on != 0;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_length(const witcert_cache* c, int layer, int* len) {
  if (witcert_status s = check_layer(c, layer)) return s;
  if (!len) return fail(WITCERT_EINVAL, "len is NULL");
  *len = c->len[layer];
  ok();
  return WITCERT_OK;
}

witcert_status witcert_seq_length(const witcert_cache* c, int layer, int seq, int* len) {
  if (witcert_status s = check_layer(c, layer)) return s;
  if (!len) return fail(WITCERT_EINVAL, "len is NULL");
  if (seq < 0 || seq >= c->cfg.batch) return fail(WITCERT_EINVAL, "sequence %d out of range [0, %d)", seq, c->cfg.batch);
  *len = c->slen[layer][seq];
  ok();
  return WITCERT_OK;
}

witcert_status witcert_export(witcert_cache* c, int layer, witcert_export_kind what, void* dst, size_t bytes,
                              void* stream) {
  if (witcert_status s = check_layer(c, layer)) return s;
  const int S = c->len[layer], nblk = (S + kBlk - 1) / kBlk;
  const size_t B = c->cfg.batch, Hkv = c->cfg.n_kv_heads, Hq = c->cfg.n_q_heads;
  size_t need = 0;
  switch (what) {
    case WITCERT_X_K_CODES: case WITCERT_X_V_CODES: need = B * S * Hkv * kD * (c->scheme == kBbox ? 2 : 1); break;
    case WITCERT_X_K_SCALES: case WITCERT_X_V_SCALES: case WITCERT_X_V_ZEROS: need = B * S * Hkv * 4 * 2; break;
    case WITCERT_X_KIVI_K_SCALE: case WITCERT_X_KIVI_K_ZERO: need = B * nblk * Hkv * kD * 2; break;
    case WITCERT_X_WITNESS: need = B * S * Hkv * kBands * 2; break;
    case WITCERT_X_SLOTS: need = B * Hkv * nblk * 4; break;
    case WITCERT_X_BLOCK_RISK: need = B * Hq * nblk * 4; break;
    case WITCERT_X_V_WITNESS: need = B * S * Hkv * 2; break;
    default: return fail(WITCERT_EINVAL, "unknown export kind %d", (int)what);
  }
  const bool int8 = int8_layout(c->scheme), kivi = c->scheme == kKivi;
  if ((what == WITCERT_X_K_SCALES && !int8) || ((what == WITCERT_X_V_SCALES) && !(int8 || kivi)) ||
      ((what == WITCERT_X_V_ZEROS || what == WITCERT_X_KIVI_K_SCALE || what == WITCERT_X_KIVI_K_ZERO) && !kivi))
    return fail(WITCERT_EINVAL, "export kind %d does not exist for this scheme", (int)what);
  if (what == WITCERT_X_BLOCK_RISK && !c->risk) return fail(WITCERT_ESTATE, "block risks need the gate enabled");
  if (what == WITCERT_X_V_WITNESS && !c->vwit) return fail(WITCERT_EINVAL, "value witnesses need a cache created with v_witness");
  if (!dst || bytes < need) return fail(WITCERT_EINVAL, "export needs %zu bytes, got %zu", need, bytes);
  auto st = static_cast<cudaStream_t>(stream);
  order_after_gate(c, layer, st);
  ExportArgs a{};
  a.blocks = c->blocks + layer * c->layer_blocks;
  a.nblk_max = c->nblk_max; a.B = (int)B; a.Hkv = (int)Hkv; a.Hq = (int)Hq; a.S = S; a.scheme = c->scheme;
  a.slots = c->slots ? c->slots + layer * layer_rows(c) * c->nblk_max : nullptr;
  a.risk = c->risk ? c->risk + (size_t)layer * B * Hq * c->nblk_max : nullptr;
  a.vwit = c->vwit ? c->vwit + layer * vwit_layer(c) : nullptr;
  a.table = c->table;
  a.dst = dst;
  a.what = (int)what;
  cudaError_t e = launch_export(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "export launch");
  c->last_write_layer = -1;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_wait_selftest(int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > 10000000000ll) return fail(WITCERT_EINVAL, "limit_ns must be in (0, 1e10]");
  int timed_out = -1;
  cudaError_t e = run_wait_selftest((uint64_t)limit_ns, static_cast<cudaStream_t>(stream), &timed_out);
  if (e != cudaSuccess) return cuda_fail(e, "wait self test");
  if (timed_out) return fail(WITCERT_ETIMEDOUT, "device wait gave up after %lld ns", (long long)limit_ns);
  ok();
  return WITCERT_OK;
}

witcert_status witcert_quotient_selftest(int n_f32, uint64_t seed, uint64_t* mismatches, void* stream) {
  if (n_f32 < 0 || n_f32 > (1 << 20) || !mismatches) return fail(WITCERT_EINVAL, "n_f32 in [0, 2^20] and a result pointer");
  unsigned long long m = 0;
  cudaError_t e = run_quotient_selftest(n_f32, seed, &m, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quotient self test");
  *mismatches = m;
  ok();
  return WITCERT_OK;
}

witcert_status witcert_dither(uint64_t seed, int layer, int kv_head, int t0, int n, int tensor, float* out,
                              void* stream) {
  if (layer < 0 || layer > 65535 || kv_head < 0 || kv_head > 65535 || t0 < 0 || n < 0 || (tensor != 0 && tensor != 1))
    return fail(WITCERT_EINVAL, "bad dither arguments");
  if (n > 0 && !out) return fail(WITCERT_EINVAL, "out is NULL");
  cudaError_t e = launch_dither(seed, layer, kv_head, t0, n, tensor, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dither launch");
  ok();
  return WITCERT_OK;
}

}  // extern "C"
