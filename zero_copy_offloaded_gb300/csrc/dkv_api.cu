// C ABI of libdkv: the host KV-cache manager, the kernel adaptor and the
// launch code.  Every compute step runs in the kernels of decode.cu,
// prefill_tc.cu, gemm_tc.cu and probes.cu; this file validates arguments, sizes the
// workspace, picks a precompiled kernel and enqueues it.
//
// KV Cache Manager ("Paper Notes: DirectKV", System Architecture): K/V live in
// pinned host memory from cudaHostAlloc, reached by the GPU through zero-copy
// pointers, written once and reused across decode iterations.
// Kernel Adaptor (same section): a lookup by (phase, dtype, head_dim, group
// size) into the instantiations compiled ahead of time, with the tile and
// stage count bounded by the shared-memory constraint
//   alpha * P >= 3 * m * size(T) * (Dim * N)
// (same page, the SMEM-capacity paragraph), alpha = 0.8 of the unified
// L1/shared pool P per SM.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>
#include <vector>

#include "dkv_internal.cuh"
#include "numa_host.h"

using namespace dkv;

namespace {

constexpr uint64_t kMagic = 0x444B5643414348ull;  // "DKVCACH"
constexpr uint64_t kDead = 0xDEADDEADDEADDEADull;

thread_local std::string g_last_error;
thread_local int g_last_launches = 0;

dkv_status fail(dkv_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
dkv_status fail(dkv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

dkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct Workspace {
  void* base = nullptr;
  size_t bytes = 0;
};

}  // namespace

namespace dkv {
// Lets the other translation units report a failure through dkv_last_error().
void set_last_error(dkv_status s, const char* msg) { fail(s, "%s", msg); }
}  // namespace dkv

struct dkv_cache {
  uint64_t magic;
  int device;
  int B, Hkv, D, max_tokens;
  dkv_dtype dtype;
  void* k_host;
  void* v_host;
  void* k_dev;
  void* v_dev;
  std::vector<int32_t> len;
  DeviceStatus* status;  // own small device allocation, never moved
  Workspace ws;
  cudaStream_t last_stream;
  int sms;
  int tune_splits, tune_tile, tune_stages;
  KernelTimer timer;      // events around the main fused kernel (measurement)
  bool timer_used;
  int debug_withhold;     // test hook for the bounded-wait path
  // paged caches (page_tokens == 0: dense [B][Hkv][max_tokens][D])
  int page_tokens, page_shift, num_pages, max_pages;
  std::vector<int32_t> pages;  // host copy of the page table [B][max_pages], -1 = none
  int* pages_dev;              // device copy read by the kernels
  // cache element format: DKV_KV_NATIVE (the dtype, 2 bytes) or DKV_KV_E4M3
  int kv_format, kv_eb;
  int numa_node_wanted, numa_node;  // host node of the GPU; node of the first cache page
  // layered caches: `layers` caches of layer_elems elements each for K and V
  int layers;
  size_t layer_elems;
  // decode-step graphs read the lengths from len_dev; set when the host
  // lengths changed outside a graph step (refreshed before the next one)
  int* len_dev;
  bool len_dev_stale;
  cudaGraphExec_t step_exec;
  cudaStream_t capture_stream;
  std::mutex mu;
};

namespace {

bool valid(const dkv_cache* c) { return c != nullptr && c->magic == kMagic; }


size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Grow the workspace to at least `need` bytes.  Growth synchronises the
// cache's last stream first so no enqueued kernel still uses the old block.
dkv_status ensure_ws(dkv_cache* c, size_t need) {
  if (c->ws.bytes >= need) return DKV_OK;
  cudaError_t e = cudaStreamSynchronize(c->last_stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  // a captured step holds addresses in the old block: it is discarded (the
  // next dkv_step_graph_launch asks for a new capture)
  if (c->step_exec) {
    cudaGraphExecDestroy(c->step_exec);
    c->step_exec = nullptr;
  }
  if (c->ws.base) cudaFree(c->ws.base);
  c->ws.base = nullptr;
  c->ws.bytes = 0;
  void* p = nullptr;
  e = cudaMalloc(&p, need);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DKV_ERR_ALLOC, "workspace cudaMalloc(%zu): %s", need, cudaGetErrorString(e));
  }
  c->ws.base = p;
  c->ws.bytes = need;
  return DKV_OK;
}

// ---- Kernel adaptor ---------------------------------------------------------
constexpr double kAlpha = 0.8;          // share of the L1/shared pool used as SMEM
constexpr double kPoolBytes = 256 * 1024;  // unified L1/shared pool per SM

bool smem_constraint_ok(int D, int N, int m, int eb) {
  return kAlpha * kPoolBytes >= 3.0 * m * (double)eb * D * N;
}

struct DecodeChoice {
  int tile_n, stages, splits, grid, smem;
};

dkv_status choose_decode(dkv_cache* c, int G, DecodeChoice* ch) {
  const int D = c->D;
  const bool fp8 = c->kv_format == DKV_KV_E4M3;
  // one 16 KB K tile + one 16 KB V tile
  int N = c->tune_tile > 0 ? c->tune_tile : 16384 / (D * c->kv_eb);
  int m = c->tune_stages > 0 ? c->tune_stages : 4;
  if ((N != 32 && N != 64 && N != 128 && N != 256) || m < 2 || m > 8)
    return fail(DKV_ERR_INVALID_ARG, "tuning tile_n=%d stages=%d out of range", N, m);
  while (m > 2 && !smem_constraint_ok(D, N, m, c->kv_eb)) --m;
  if (!smem_constraint_ok(D, N, m, c->kv_eb))
    return fail(DKV_ERR_UNSUPPORTED, "tile %d x %d fails the shared-memory constraint", N, D);
  if (fp8 && N * G < 256 && (D / (256 / (N * G))) % 16 != 0)
    return fail(DKV_ERR_UNSUPPORTED, "tile %d: an E4M3 score slice must span whole 16-byte chunks", N);
  const int smem = decode_smem_bytes(c->dtype, D, G, N, m, c->B, fp8);
  int occ = 0;
  cudaError_t e = decode_occupancy(c->dtype, D, G, N, m, c->B, &occ, fp8);
  if (e != cudaSuccess) return cuda_fail(e, "decode occupancy");
  if (occ < 1) return fail(DKV_ERR_UNSUPPORTED, "decode kernel does not fit on an SM (smem %d)", smem);
  const int grid = c->sms * occ;
  // splits: minimise the most tiles any CTA streams (units go round-robin)
  int splits = c->tune_splits;
  if (splits <= 0) {
    int maxS = 1;
    for (int b = 0; b < c->B; ++b) maxS = std::max(maxS, c->len[b] + 1);
    const int nt = (maxS + N - 1) / N;
    const int bh = c->B * c->Hkv;
    long best = -1;
    splits = 1;
    for (int s = 1; s <= std::min(nt, 1024); ++s) {
      const long units = (long)bh * s;
      const long waves = (units + grid - 1) / grid;
      const long per_unit = (nt + s - 1) / s;
      const long cost = waves * per_unit * 64 + waves;  // tiles, plus a little per unit
      if (best < 0 || cost < best) { best = cost; splits = s; }
    }
  }
  ch->tile_n = N;
  ch->stages = m;
  ch->splits = splits;
  ch->grid = grid;
  ch->smem = smem;
  return DKV_OK;
}

dkv_status check_call(dkv_cache* c, const void* x, const void* wq, const void* wk,
                      const void* wv, int hidden, int n_q_heads, const void* out, int T) {
  if (!valid(c)) return fail(DKV_ERR_INVALID_ARG, "invalid cache handle");
  if (!x || !wq || !wk || !wv || !out) return fail(DKV_ERR_INVALID_ARG, "null tensor pointer");
  if (hidden <= 0 || hidden % 16 != 0)
    return fail(DKV_ERR_INVALID_ARG, "hidden=%d must be a positive multiple of 16", hidden);
  if (n_q_heads <= 0 || n_q_heads % c->Hkv != 0)
    return fail(DKV_ERR_INVALID_ARG, "n_q_heads=%d must be a positive multiple of Hkv=%d",
                n_q_heads, c->Hkv);
  if (T <= 0) return fail(DKV_ERR_INVALID_ARG, "T=%d must be positive", T);
  for (int b = 0; b < c->B; ++b)
    if ((long)c->len[b] + T > c->max_tokens)
      return fail(DKV_ERR_CAPACITY, "sequence %d: length %d + %d new > max_tokens %d", b,
                  c->len[b], T, c->max_tokens);
  if (c->page_tokens) {
    // every row the call reads or writes, [0, len + T), must sit on a page
    for (int b = 0; b < c->B; ++b) {
      const int need = (c->len[b] + T + c->page_tokens - 1) >> c->page_shift;
      for (int i = 0; i < need; ++i)
        if (c->pages[(size_t)b * c->max_pages + i] < 0)
          return fail(DKV_ERR_CAPACITY, "sequence %d: logical page %d (of %d needed) has no page",
                      b, i, need);
    }
  }
  return DKV_OK;
}

size_t pool_rows(const dkv_cache* c) {
  return c->page_tokens ? (size_t)c->num_pages * c->Hkv * c->page_tokens
                        : (size_t)c->B * c->Hkv * c->max_tokens;
}

CacheLayout layout_of(const dkv_cache* c) {
  CacheLayout l;
  l.pages = c->page_tokens ? c->pages_dev : nullptr;
  l.page_shift = c->page_shift;
  l.max_pages = c->max_pages;
  l.Hkv = c->Hkv;
  l.S_max = c->max_tokens;
  return l;
}

void fill_lens(int* dst, const std::vector<int32_t>& len) {
  for (int b = 0; b < kMaxBatch; ++b) dst[b] = b < (int)len.size() ? len[b] : 0;
}

dkv_status set_device(dkv_cache* c) {
  cudaError_t e = cudaSetDevice(c->device);
  return e == cudaSuccess ? DKV_OK : cuda_fail(e, "cudaSetDevice");
}

// Shared by dkv_decode, dkv_decode_staged and dkv_decode_unfused.
dkv_status decode_impl(dkv_cache* c, const void* x, const void* wq, const void* wk,
                       const void* wv, int hidden, int n_q_heads, void* out,
                       const void* k_read, const void* v_read, cudaStream_t s,
                       bool unfused = false, int layer = 0, bool capture = false) {
  const int G = n_q_heads / c->Hkv;
  if (!decode_supported(c->dtype, c->D, G))
    return fail(DKV_ERR_UNSUPPORTED, "no decode kernel for dtype=%d D=%d G=%d", c->dtype, c->D, G);
  DecodeChoice ch;
  dkv_status st = choose_decode(c, G, &ch);
  if (st != DKV_OK) return st;
  const int B = c->B, D = c->D, Hq = n_q_heads;
  const size_t q_b = align_up((size_t)B * Hq * D * 2, 256);
  const size_t kv_b = align_up((size_t)B * 2 * c->Hkv * D * 2, 256);
  const size_t po_b = align_up((size_t)B * Hq * ch.splits * D * 4, 256);
  const size_t pl_b = align_up((size_t)B * Hq * ch.splits * 4, 256);
  st = ensure_ws(c, q_b + kv_b + po_b + pl_b);
  if (st != DKV_OK) return st;
  DecodeParams p;
  memset(&p, 0, sizeof p);
  char* w = static_cast<char*>(c->ws.base);
  p.x = x; p.wq = wq; p.wk = wk; p.wv = wv;
  const size_t loff = (size_t)layer * c->layer_elems * c->kv_eb;  // bytes
  p.k_read = static_cast<const char*>(k_read) + loff;
  p.v_read = static_cast<const char*>(v_read) + loff;
  p.k_host = static_cast<char*>(c->k_dev) + loff;
  p.v_host = static_cast<char*>(c->v_dev) + loff;
  p.q_ws = w; p.kv_ws = w + q_b;
  p.part_o = reinterpret_cast<float*>(w + q_b + kv_b);
  p.part_lse = reinterpret_cast<float*>(w + q_b + kv_b + po_b);
  p.status = c->status;
  p.out = out;
  p.B = B; p.H = hidden; p.Hq = Hq; p.Hkv = c->Hkv; p.D = D; p.S_max = c->max_tokens;
  p.splits = ch.splits; p.tile_n = ch.tile_n; p.stages = ch.stages;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  p.debug_withhold = c->debug_withhold;
  p.lay = layout_of(c);
  p.kv_fp8 = c->kv_format == DKV_KV_E4M3;
  fill_lens(p.len, c->len);
  if (capture) p.len_dev = c->len_dev;
  if (!capture) g_last_launches = 0;
  cudaError_t e;
  if (unfused) {  // projection + append, then attention over host rows only
    p.mode = kDecodeProjectOnly;
    e = launch_decode(p, c->dtype, ch.grid, ch.smem, s, &g_last_launches, KernelTimer());
    p.mode = kDecodeAttendOnly;
    if (e == cudaSuccess)
      e = launch_decode(p, c->dtype, ch.grid, ch.smem, s, &g_last_launches, c->timer);
  } else {
    e = launch_decode(p, c->dtype, ch.grid, ch.smem, s, &g_last_launches,
                      capture ? KernelTimer() : c->timer);
  }
  if (capture) return e == cudaSuccess ? DKV_OK : cuda_fail(e, "decode launch in a capture");
  c->timer_used = c->timer.start != nullptr;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "decode launch");
  }
  c->last_stream = s;
  if (layer == c->layers - 1) {  // a token is complete once its last layer is
    for (int b = 0; b < B; ++b) c->len[b] += 1;
    c->len_dev_stale = true;
  }
  return DKV_OK;
}

// Workspace bytes a decode call with G query heads per KV head needs.
size_t decode_ws_bytes(const dkv_cache* c, int n_q_heads, int splits) {
  const int B = c->B, D = c->D;
  return align_up((size_t)B * n_q_heads * D * 2, 256) + align_up((size_t)B * 2 * c->Hkv * D * 2, 256) +
         align_up((size_t)B * n_q_heads * splits * D * 4, 256) +
         align_up((size_t)B * n_q_heads * splits * 4, 256);
}

}  // namespace

extern "C" {

const char* dkv_status_str(dkv_status s) {
  switch (s) {
    case DKV_OK: return "ok";
    case DKV_ERR_INVALID_ARG: return "invalid argument";
    case DKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case DKV_ERR_CAPACITY: return "cache capacity exceeded";
    case DKV_ERR_NO_MAPPED_MEMORY: return "device cannot map host memory";
    case DKV_ERR_ALLOC: return "allocation failed";
    case DKV_ERR_CUDA: return "CUDA error";
    case DKV_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* dkv_last_error(void) { return g_last_error.c_str(); }

int dkv_last_launch_count(void) { return g_last_launches; }

// Shared by the dense and the paged allocation: `rows` cache rows of D
// elements each for K and for V in pinned, mapped host memory.
static dkv_status alloc_common(dkv_cache** out, int batch, int n_kv_heads, int head_dim,
                               int max_tokens, dkv_dtype dtype, size_t rows, int page_tokens,
                               int num_pages, int max_pages, int layers = 1,
                               int kv_format = DKV_KV_NATIVE) {
  if (!out) return fail(DKV_ERR_INVALID_ARG, "null output handle");
  *out = nullptr;
  if (batch <= 0 || batch > kMaxBatch)
    return fail(DKV_ERR_INVALID_ARG, "batch=%d must be in [1, %d]", batch, kMaxBatch);
  if (n_kv_heads <= 0 || max_tokens <= 0)
    return fail(DKV_ERR_INVALID_ARG, "n_kv_heads=%d and max_tokens=%d must be positive",
                n_kv_heads, max_tokens);
  if (dtype != DKV_BF16 && dtype != DKV_FP16)
    return fail(DKV_ERR_INVALID_ARG, "dtype=%d is not bf16 (0) or fp16 (1)", (int)dtype);
  if (head_dim != 64 && head_dim != 128)
    return fail(DKV_ERR_UNSUPPORTED, "head_dim=%d (supported: 64, 128)", head_dim);
  // Host-side fault injection for tests: the allocation reports failure
  // without touching the GPU.
  const char* inject = getenv("DKV_FAULT_INJECT");
  if (inject && strcmp(inject, "host_alloc") == 0)
    return fail(DKV_ERR_ALLOC, "cudaHostAlloc failed (injected on the host)");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int can_map = 0, sms = 0;
  cudaDeviceGetAttribute(&can_map, cudaDevAttrCanMapHostMemory, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (!can_map) return fail(DKV_ERR_NO_MAPPED_MEMORY, "device %d cannot map host memory", dev);
  if (kv_format != DKV_KV_NATIVE && kv_format != DKV_KV_E4M3)
    return fail(DKV_ERR_INVALID_ARG, "kv_format=%d is not native (0) or E4M3 (1)", kv_format);
  if (kv_format == DKV_KV_E4M3 && dtype != DKV_BF16)
    return fail(DKV_ERR_UNSUPPORTED, "E4M3 caches take bf16 activations");
  const int kv_eb = kv_format == DKV_KV_E4M3 ? 1 : 2;
  const size_t bytes = rows * head_dim * kv_eb * layers;
  void* kh = nullptr;
  void* vh = nullptr;
  // pinned on the host NUMA node attached to this GPU, where known
  const int node = device_numa_node(dev);
  {
    NumaScope scope(node);
    e = cudaHostAlloc(&kh, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(DKV_ERR_ALLOC, "cudaHostAlloc(%zu) for K: %s", bytes, cudaGetErrorString(e));
    }
    e = cudaHostAlloc(&vh, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
      cudaGetLastError();
      cudaFreeHost(kh);
      return fail(DKV_ERR_ALLOC, "cudaHostAlloc(%zu) for V: %s", bytes, cudaGetErrorString(e));
    }
    memset(kh, 0, bytes);
    memset(vh, 0, bytes);
  }
  void* kd = nullptr;
  void* vd = nullptr;
  if ((e = cudaHostGetDevicePointer(&kd, kh, 0)) != cudaSuccess ||
      (e = cudaHostGetDevicePointer(&vd, vh, 0)) != cudaSuccess) {
    cudaGetLastError();
    cudaFreeHost(kh);
    cudaFreeHost(vh);
    return cuda_fail(e, "cudaHostGetDevicePointer");
  }
  DeviceStatus* st = nullptr;
  if ((e = cudaMalloc(&st, sizeof(DeviceStatus))) != cudaSuccess) {
    cudaGetLastError();
    cudaFreeHost(kh);
    cudaFreeHost(vh);
    return fail(DKV_ERR_ALLOC, "status cudaMalloc: %s", cudaGetErrorString(e));
  }
  int* pages_dev = nullptr;
  const size_t table = (size_t)batch * max_pages;
  if (page_tokens) {
    if ((e = cudaMalloc(&pages_dev, table * sizeof(int32_t))) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(st);
      cudaFreeHost(kh);
      cudaFreeHost(vh);
      return fail(DKV_ERR_ALLOC, "page table cudaMalloc: %s", cudaGetErrorString(e));
    }
    cudaMemset(pages_dev, 0xff, table * sizeof(int32_t));  // -1: no page
  }
  int* len_dev = nullptr;
  if ((e = cudaMalloc(&len_dev, kMaxBatch * sizeof(int))) != cudaSuccess) {
    cudaGetLastError();
    if (pages_dev) cudaFree(pages_dev);
    cudaFree(st);
    cudaFreeHost(kh);
    cudaFreeHost(vh);
    return fail(DKV_ERR_ALLOC, "lengths cudaMalloc: %s", cudaGetErrorString(e));
  }
  cudaMemset(len_dev, 0, kMaxBatch * sizeof(int));
  cudaMemset(st, 0, sizeof(DeviceStatus));
  cudaDeviceSynchronize();
  dkv_cache* c = new dkv_cache;
  c->magic = kMagic;
  c->device = dev;
  c->B = batch; c->Hkv = n_kv_heads; c->D = head_dim; c->max_tokens = max_tokens;
  c->dtype = dtype;
  c->k_host = kh; c->v_host = vh; c->k_dev = kd; c->v_dev = vd;
  c->len.assign(batch, 0);
  c->status = st;
  c->last_stream = nullptr;
  c->sms = sms;
  c->tune_splits = c->tune_tile = c->tune_stages = 0;
  c->timer_used = false;
  c->debug_withhold = 0;
  c->page_tokens = page_tokens;
  c->page_shift = 0;
  while (page_tokens && (1 << c->page_shift) < page_tokens) ++c->page_shift;
  c->num_pages = num_pages;
  c->max_pages = max_pages;
  c->pages.assign(table, -1);
  c->pages_dev = pages_dev;
  c->layers = layers;
  c->layer_elems = rows * head_dim;
  c->kv_format = kv_format;
  c->kv_eb = kv_eb;
  c->numa_node_wanted = node;
  c->numa_node = page_numa_node(kh);
  c->len_dev = len_dev;
  c->len_dev_stale = false;
  c->step_exec = nullptr;
  c->capture_stream = nullptr;
  *out = c;
  return DKV_OK;
}

dkv_status dkv_cache_alloc_layered(dkv_cache** out, int layers, int batch, int n_kv_heads,
                                   int head_dim, int max_tokens, dkv_dtype dtype) {
  if (!out) return fail(DKV_ERR_INVALID_ARG, "null output handle");
  *out = nullptr;
  if (layers <= 0 || layers > 1024)
    return fail(DKV_ERR_INVALID_ARG, "layers=%d must be in [1, 1024]", layers);
  if (batch <= 0 || batch > kMaxBatch)
    return fail(DKV_ERR_INVALID_ARG, "batch=%d must be in [1, %d]", batch, kMaxBatch);
  if (n_kv_heads <= 0 || max_tokens <= 0)
    return fail(DKV_ERR_INVALID_ARG, "n_kv_heads=%d and max_tokens=%d must be positive",
                n_kv_heads, max_tokens);
  return alloc_common(out, batch, n_kv_heads, head_dim, max_tokens, dtype,
                      (size_t)batch * n_kv_heads * max_tokens, 0, 0, 0, layers);
}

dkv_status dkv_cache_alloc(dkv_cache** out, int batch, int n_kv_heads, int head_dim,
                           int max_tokens, dkv_dtype dtype) {
  if (!out) return fail(DKV_ERR_INVALID_ARG, "null output handle");
  *out = nullptr;
  if (batch <= 0 || batch > kMaxBatch)
    return fail(DKV_ERR_INVALID_ARG, "batch=%d must be in [1, %d]", batch, kMaxBatch);
  if (n_kv_heads <= 0 || max_tokens <= 0)
    return fail(DKV_ERR_INVALID_ARG, "n_kv_heads=%d and max_tokens=%d must be positive",
                n_kv_heads, max_tokens);
  return alloc_common(out, batch, n_kv_heads, head_dim, max_tokens, dtype,
                      (size_t)batch * n_kv_heads * max_tokens, 0, 0, 0);
}

dkv_status dkv_cache_alloc_ex(dkv_cache** out, const dkv_cache_desc_t* d) {
  if (!out) return fail(DKV_ERR_INVALID_ARG, "null output handle");
  *out = nullptr;
  if (!d) return fail(DKV_ERR_INVALID_ARG, "null description");
  const int layers = d->layers > 0 ? d->layers : 1;
  if (layers > 1024) return fail(DKV_ERR_INVALID_ARG, "layers=%d must be in [1, 1024]", layers);
  if (d->batch <= 0 || d->batch > kMaxBatch)
    return fail(DKV_ERR_INVALID_ARG, "batch=%d must be in [1, %d]", d->batch, kMaxBatch);
  if (d->n_kv_heads <= 0)
    return fail(DKV_ERR_INVALID_ARG, "n_kv_heads=%d must be positive", d->n_kv_heads);
  if (d->page_tokens) {
    if (layers != 1) return fail(DKV_ERR_UNSUPPORTED, "paged caches hold one layer");
    if (d->page_tokens < 1 || d->page_tokens > 4096 || (d->page_tokens & (d->page_tokens - 1)))
      return fail(DKV_ERR_INVALID_ARG, "page_tokens=%d must be a power of two in [1, 4096]",
                  d->page_tokens);
    if (d->num_pages <= 0 || d->max_pages_per_seq <= 0)
      return fail(DKV_ERR_INVALID_ARG, "num_pages and max_pages_per_seq must be positive");
    if ((long long)d->max_pages_per_seq * d->page_tokens > (1LL << 30))
      return fail(DKV_ERR_INVALID_ARG, "max_pages_per_seq * page_tokens is too large");
    return alloc_common(out, d->batch, d->n_kv_heads, d->head_dim,
                        d->max_pages_per_seq * d->page_tokens, d->dtype,
                        (size_t)d->num_pages * d->n_kv_heads * d->page_tokens, d->page_tokens,
                        d->num_pages, d->max_pages_per_seq, 1, d->kv_format);
  }
  if (d->max_tokens <= 0) return fail(DKV_ERR_INVALID_ARG, "max_tokens=%d must be positive", d->max_tokens);
  return alloc_common(out, d->batch, d->n_kv_heads, d->head_dim, d->max_tokens, d->dtype,
                      (size_t)d->batch * d->n_kv_heads * d->max_tokens, 0, 0, 0, layers,
                      d->kv_format);
}

dkv_status dkv_cache_alloc_paged(dkv_cache** out, int batch, int n_kv_heads, int head_dim,
                                 int page_tokens, int num_pages, int max_pages_per_seq,
                                 dkv_dtype dtype) {
  if (!out) return fail(DKV_ERR_INVALID_ARG, "null output handle");
  *out = nullptr;
  if (batch <= 0 || batch > kMaxBatch)
    return fail(DKV_ERR_INVALID_ARG, "batch=%d must be in [1, %d]", batch, kMaxBatch);
  if (n_kv_heads <= 0 || num_pages <= 0 || max_pages_per_seq <= 0)
    return fail(DKV_ERR_INVALID_ARG, "n_kv_heads=%d, num_pages=%d and max_pages_per_seq=%d "
                "must be positive", n_kv_heads, num_pages, max_pages_per_seq);
  if (page_tokens < 1 || page_tokens > 4096 || (page_tokens & (page_tokens - 1)))
    return fail(DKV_ERR_INVALID_ARG, "page_tokens=%d must be a power of two in [1, 4096]",
                page_tokens);
  if ((long long)max_pages_per_seq * page_tokens > (1LL << 30))
    return fail(DKV_ERR_INVALID_ARG, "max_pages_per_seq * page_tokens is too large");
  return alloc_common(out, batch, n_kv_heads, head_dim, max_pages_per_seq * page_tokens, dtype,
                      (size_t)num_pages * n_kv_heads * page_tokens, page_tokens, num_pages,
                      max_pages_per_seq);
}

dkv_status dkv_cache_set_page_table(dkv_cache* c, const int32_t* table) {
  if (!valid(c) || !table) return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  if (!c->page_tokens) return fail(DKV_ERR_INVALID_ARG, "the cache is dense, not paged");
  const size_t n = c->pages.size();
  for (size_t i = 0; i < n; ++i)
    if (table[i] < -1 || table[i] >= c->num_pages)
      return fail(DKV_ERR_INVALID_ARG, "page table entry %zu = %d outside [-1, %d)", i, table[i],
                  c->num_pages);
  std::lock_guard<std::mutex> lk(c->mu);
  dkv_status st = set_device(c);
  if (st != DKV_OK) return st;
  // enqueued calls may still read the previous table
  cudaError_t e = cudaStreamSynchronize(c->last_stream);
  if (e == cudaSuccess)
    e = cudaMemcpy(c->pages_dev, table, n * sizeof(int32_t), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "page table copy");
  c->pages.assign(table, table + n);
  return DKV_OK;
}



dkv_status dkv_free(dkv_cache* c) {
  if (!valid(c)) return fail(DKV_ERR_INVALID_ARG, "invalid or already freed cache handle");
  c->magic = kDead;
  cudaSetDevice(c->device);
  cudaDeviceSynchronize();
  if (c->ws.base) cudaFree(c->ws.base);
  if (c->timer.start) cudaEventDestroy(c->timer.start);
  if (c->timer.stop) cudaEventDestroy(c->timer.stop);
  c->timer = KernelTimer();
  cudaFree(c->status);
  if (c->pages_dev) cudaFree(c->pages_dev);
  c->pages_dev = nullptr;
  if (c->len_dev) cudaFree(c->len_dev);
  c->len_dev = nullptr;
  if (c->step_exec) cudaGraphExecDestroy(c->step_exec);
  c->step_exec = nullptr;
  if (c->capture_stream) cudaStreamDestroy(c->capture_stream);
  c->capture_stream = nullptr;
  cudaFreeHost(c->k_host);
  cudaFreeHost(c->v_host);
  // The handle memory is kept (tagged dead) so a second free is detected
  // instead of touching freed memory.
  c->ws.base = nullptr;
  c->k_host = c->v_host = c->k_dev = c->v_dev = nullptr;
  return DKV_OK;
}

dkv_status dkv_cache_host_ptrs(dkv_cache* c, void** k, void** v) {
  if (!valid(c) || !k || !v) return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  *k = c->k_host;
  *v = c->v_host;
  return DKV_OK;
}

dkv_status dkv_cache_device_ptrs(dkv_cache* c, void** k, void** v) {
  if (!valid(c) || !k || !v) return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  *k = c->k_dev;
  *v = c->v_dev;
  return DKV_OK;
}

dkv_status dkv_cache_set_lengths(dkv_cache* c, const int32_t* len) {
  if (!valid(c) || !len) return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  for (int b = 0; b < c->B; ++b) {
    if (len[b] < 0) return fail(DKV_ERR_INVALID_ARG, "length %d of sequence %d", len[b], b);
    if (len[b] > c->max_tokens)
      return fail(DKV_ERR_CAPACITY, "length %d of sequence %d > max_tokens %d", len[b], b,
                  c->max_tokens);
  }
  for (int b = 0; b < c->B; ++b) c->len[b] = len[b];
  c->len_dev_stale = true;
  return DKV_OK;
}

dkv_status dkv_cache_get_lengths(const dkv_cache* c, int32_t* len) {
  if (!valid(c) || !len) return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  for (int b = 0; b < c->B; ++b) len[b] = c->len[b];
  return DKV_OK;
}

dkv_status dkv_cache_info(const dkv_cache* c, dkv_cache_info_t* info) {
  if (!valid(c) || !info) return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  info->host_pinned_bytes = 2 * pool_rows(c) * c->D * c->kv_eb * c->layers;
  info->device_workspace_bytes = c->ws.bytes + sizeof(DeviceStatus) +
                                 c->pages.size() * sizeof(int32_t);
  info->device_staging_bytes = 0;
  info->batch = c->B; info->n_kv_heads = c->Hkv; info->head_dim = c->D;
  info->max_tokens = c->max_tokens; info->dtype = c->dtype;
  info->page_tokens = c->page_tokens; info->num_pages = c->num_pages;
  info->max_pages_per_seq = c->max_pages;
  info->layers = c->layers;
  info->kv_format = c->kv_format;
  info->numa_node_wanted = c->numa_node_wanted;
  info->numa_node = c->numa_node;
  return DKV_OK;
}

dkv_status dkv_cache_debug_withhold(dkv_cache* c, int enable) {
  if (!valid(c)) return fail(DKV_ERR_INVALID_ARG, "invalid cache handle");
  c->debug_withhold = enable ? 1 : 0;
  return DKV_OK;
}

dkv_status dkv_cache_set_tuning(dkv_cache* c, int splits, int tile_n, int stages) {
  if (!valid(c)) return fail(DKV_ERR_INVALID_ARG, "invalid cache handle");
  if (splits < 0 || tile_n < 0 || stages < 0)
    return fail(DKV_ERR_INVALID_ARG, "negative tuning value");
  c->tune_splits = splits;
  c->tune_tile = tile_n;
  c->tune_stages = stages;
  return DKV_OK;
}

dkv_status dkv_cache_reserve(dkv_cache* c, int n_q_heads, int max_new_tokens) {
  if (!valid(c) || n_q_heads <= 0 || max_new_tokens <= 0 || n_q_heads % c->Hkv)
    return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  std::lock_guard<std::mutex> lk(c->mu);
  dkv_status st = set_device(c);
  if (st != DKV_OK) return st;
  const int D = c->D, B = c->B, Hq = n_q_heads, T = max_new_tokens;
  // decode: worst case of the split search is bounded by the tile count
  const int G = Hq / c->Hkv;
  size_t need = 0;
  if (decode_supported(c->dtype, D, G)) {
    const int N = 8192 / D;
    const int nt = (c->max_tokens + N - 1) / N;
    const size_t splits = std::min(nt, 1024);
    need = align_up((size_t)B * Hq * D * 2, 256) + align_up((size_t)B * 2 * c->Hkv * D * 2, 256) +
           align_up((size_t)B * Hq * splits * D * 4, 256) + align_up((size_t)B * Hq * splits * 4, 256);
  }
  const int C = prefill_tc_chunk_keys();
  const size_t nch = (size_t)(c->max_tokens + C - 1) / C;
  const size_t rows = (size_t)B * T * Hq;
  const size_t pre = align_up(rows * D * 2, 256) + align_up(nch * rows * D * 2, 256) +
                     align_up(nch * rows * 4, 256) + align_up(nch * B * c->Hkv * 4, 256);
  return ensure_ws(c, std::max(need, pre));
}

dkv_status dkv_decode_layer(dkv_cache* c, int layer, const void* x, const void* wq,
                            const void* wk, const void* wv, int hidden, int n_q_heads, void* out,
                            void* stream) {
  dkv_status st = check_call(c, x, wq, wk, wv, hidden, n_q_heads, out, 1);
  if (st != DKV_OK) return st;
  if (layer < 0 || layer >= c->layers)
    return fail(DKV_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, c->layers);
  std::lock_guard<std::mutex> lk(c->mu);
  if ((st = set_device(c)) != DKV_OK) return st;
  return decode_impl(c, x, wq, wk, wv, hidden, n_q_heads, out, c->k_dev, c->v_dev,
                     static_cast<cudaStream_t>(stream), false, layer);
}

dkv_status dkv_decode(dkv_cache* c, const void* x, const void* wq, const void* wk,
                      const void* wv, int hidden, int n_q_heads, void* out, void* stream) {
  if (valid(c) && c->layers != 1)
    return fail(DKV_ERR_INVALID_ARG, "a layered cache takes dkv_decode_layer");
  return dkv_decode_layer(c, 0, x, wq, wk, wv, hidden, n_q_heads, out, stream);
}

dkv_status dkv_step_graph_capture(dkv_cache* c, int hidden, int n_q_heads,
                                  const void* const* x, const void* const* wq,
                                  const void* const* wk, const void* const* wv,
                                  void* const* out) {
  if (!valid(c) || !x || !wq || !wk || !wv || !out)
    return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  for (int l = 0; l < c->layers; ++l) {
    dkv_status st = check_call(c, x[l], wq[l], wk[l], wv[l], hidden, n_q_heads, out[l], 1);
    if (st != DKV_OK) return st;
  }
  std::lock_guard<std::mutex> lk(c->mu);
  dkv_status st = set_device(c);
  if (st != DKV_OK) return st;
  const int G = n_q_heads / c->Hkv;
  if (!decode_supported(c->dtype, c->D, G))
    return fail(DKV_ERR_UNSUPPORTED, "no decode kernel for dtype=%d D=%d G=%d", c->dtype, c->D, G);
  DecodeChoice ch;
  if ((st = choose_decode(c, G, &ch)) != DKV_OK) return st;
  // everything a capture must not do: allocate, synchronise
  if ((st = ensure_ws(c, decode_ws_bytes(c, n_q_heads, ch.splits))) != DKV_OK) return st;
  cudaError_t e = cudaSuccess;
  if (!c->capture_stream) e = cudaStreamCreateWithFlags(&c->capture_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->last_stream);
  if (e != cudaSuccess) return cuda_fail(e, "capture stream");
  if (c->step_exec) cudaGraphExecDestroy(c->step_exec);
  c->step_exec = nullptr;
  cudaStream_t cs = c->capture_stream;
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamBeginCapture");
  g_last_launches = 0;
  for (int l = 0; l < c->layers && st == DKV_OK; ++l)
    st = decode_impl(c, x[l], wq[l], wk[l], wv[l], hidden, n_q_heads, out[l], c->k_dev, c->v_dev,
                     cs, false, l, true);
  if (st == DKV_OK) {
    e = launch_advance_lengths(c->len_dev, c->B, 1, cs);
    if (e != cudaSuccess) st = cuda_fail(e, "length update in a capture");
  }
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(cs, &graph);
  if (st != DKV_OK) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return st;
  }
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
  e = cudaGraphInstantiate(&c->step_exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) {
    c->step_exec = nullptr;
    return cuda_fail(e, "cudaGraphInstantiate");
  }
  c->len_dev_stale = true;  // written from the host lengths before the first launch
  return DKV_OK;
}

dkv_status dkv_step_graph_launch(dkv_cache* c, void* stream) {
  if (!valid(c)) return fail(DKV_ERR_INVALID_ARG, "invalid cache handle");
  if (!c->step_exec) return fail(DKV_ERR_INVALID_ARG, "no decode step has been captured");
  for (int b = 0; b < c->B; ++b)
    if ((long)c->len[b] + 1 > c->max_tokens)
      return fail(DKV_ERR_CAPACITY, "sequence %d: length %d + 1 > max_tokens %d", b, c->len[b],
                  c->max_tokens);
  std::lock_guard<std::mutex> lk(c->mu);
  dkv_status st = set_device(c);
  if (st != DKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (c->len_dev_stale) {  // lengths changed outside graph steps: publish them first
    e = cudaStreamSynchronize(c->last_stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess)
      e = cudaMemcpy(c->len_dev, c->len.data(), c->B * sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "lengths copy");
    c->len_dev_stale = false;
  }
  e = cudaGraphLaunch(c->step_exec, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
  c->last_stream = s;
  for (int b = 0; b < c->B; ++b) c->len[b] += 1;
  return DKV_OK;
}

dkv_status dkv_decode_unfused(dkv_cache* c, const void* x, const void* wq, const void* wk,
                              const void* wv, int hidden, int n_q_heads, void* out, void* stream) {
  dkv_status st = check_call(c, x, wq, wk, wv, hidden, n_q_heads, out, 1);
  if (st != DKV_OK) return st;
  if (c->layers != 1) return fail(DKV_ERR_UNSUPPORTED, "unfused decode needs a one-layer cache");
  std::lock_guard<std::mutex> lk(c->mu);
  if ((st = set_device(c)) != DKV_OK) return st;
  return decode_impl(c, x, wq, wk, wv, hidden, n_q_heads, out, c->k_dev, c->v_dev,
                     static_cast<cudaStream_t>(stream), true);
}

dkv_status dkv_decode_staged(dkv_cache* c, const void* x, const void* wq, const void* wk,
                             const void* wv, int hidden, int n_q_heads, void* out,
                             void* k_stage, void* v_stage, void* stream) {
  dkv_status st = check_call(c, x, wq, wk, wv, hidden, n_q_heads, out, 1);
  if (st != DKV_OK) return st;
  if (!k_stage || !v_stage) return fail(DKV_ERR_INVALID_ARG, "null staging buffer");
  if (c->page_tokens || c->layers != 1 || c->kv_format != DKV_KV_NATIVE)
    return fail(DKV_ERR_UNSUPPORTED, "staged decode needs a dense one-layer 16-bit cache");
  std::lock_guard<std::mutex> lk(c->mu);
  if ((st = set_device(c)) != DKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t head_elems = (size_t)c->max_tokens * c->D;
  for (int b = 0; b < c->B; ++b)
    for (int h = 0; h < c->Hkv; ++h) {
      const size_t off = ((size_t)b * c->Hkv + h) * head_elems * 2;
      const size_t n = (size_t)c->len[b] * c->D * 2;
      if (n == 0) continue;
      cudaError_t e = cudaMemcpyAsync(static_cast<char*>(k_stage) + off,
                                      static_cast<char*>(c->k_host) + off, n,
                                      cudaMemcpyHostToDevice, s);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(static_cast<char*>(v_stage) + off,
                            static_cast<char*>(c->v_host) + off, n, cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) return cuda_fail(e, "staging cudaMemcpyAsync");
    }
  return decode_impl(c, x, wq, wk, wv, hidden, n_q_heads, out, k_stage, v_stage, s);
}

namespace {

// Shared by dkv_prefill_layer and dkv_prefill_staged: the cached rows are read
// from k_read / v_read (the host cache, or an HBM copy of it), the new rows
// are appended to the host cache.  Called with the cache's mutex held.
dkv_status prefill_impl(dkv_cache* c, int layer, const void* x, int T, const void* wq,
                        const void* wk, const void* wv, int hidden, int n_q_heads, void* out,
                        const void* k_read, const void* v_read, void* stream,
                        bool naive = false) {
  dkv_status st;
  const int G = n_q_heads / c->Hkv;
  if (!prefill_supported(c->dtype, c->D, G))
    return fail(DKV_ERR_UNSUPPORTED, "no prefill kernel for dtype=%d D=%d G=%d", c->dtype, c->D, G);
  const int B = c->B, D = c->D, Hq = n_q_heads;
  const int C = prefill_tc_chunk_keys();
  int maxS = 0;
  for (int b = 0; b < B; ++b) maxS = std::max(maxS, c->len[b] + T);
  const int nchunks = (maxS + C - 1) / C;
  const size_t rows = (size_t)B * T * Hq;
  const size_t q_b = align_up(rows * D * 2, 256);
  const size_t po_b = align_up((size_t)nchunks * rows * D * 2, 256);  // partials in the dtype
  const size_t pl_b = align_up((size_t)nchunks * rows * 4, 256);
  const size_t pk_b = align_up((size_t)nchunks * B * c->Hkv * 4, 256);
  if ((st = ensure_ws(c, q_b + po_b + pl_b + pk_b)) != DKV_OK) return st;
  char* w = static_cast<char*>(c->ws.base);
  PrefillParams p;
  memset(&p, 0, sizeof p);
  p.x = x; p.wk = wk; p.wv = wv; p.q = w;
  const size_t loff = (size_t)layer * c->layer_elems * c->kv_eb;  // bytes
  p.k_read = static_cast<const char*>(k_read) + loff;
  p.v_read = static_cast<const char*>(v_read) + loff;
  p.k_host = static_cast<char*>(c->k_dev) + loff;
  p.v_host = static_cast<char*>(c->v_dev) + loff;
  p.part_o = w + q_b;
  p.part_lse = reinterpret_cast<float*>(w + q_b + po_b);
  p.part_k = reinterpret_cast<int*>(w + q_b + po_b + pl_b);
  p.status = c->status;
  p.out = out;
  p.B = B; p.T = T; p.H = hidden; p.Hq = Hq; p.Hkv = c->Hkv; p.D = D; p.S_max = c->max_tokens;
  p.chunk = C; p.nchunks = nchunks;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  p.lay = layout_of(c);
  p.naive = naive ? 1 : 0;
  p.debug_withhold = c->debug_withhold;
  p.kv_fp8 = c->kv_format == DKV_KV_E4M3;
  fill_lens(p.len, c->len);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  g_last_launches = 0;
  cudaError_t e = launch_prefill_tc(p, c->dtype, wq, s, &g_last_launches, c->timer);
  c->timer_used = c->timer.start != nullptr;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "prefill launch");
  }
  c->last_stream = s;
  if (layer == c->layers - 1) {  // the tokens are complete once their last layer is
    for (int b = 0; b < B; ++b) c->len[b] += T;
    c->len_dev_stale = true;
  }
  return DKV_OK;
}

}  // namespace

dkv_status dkv_prefill_layer(dkv_cache* c, int layer, const void* x, int T, const void* wq,
                             const void* wk, const void* wv, int hidden, int n_q_heads, void* out,
                             void* stream) {
  dkv_status st = check_call(c, x, wq, wk, wv, hidden, n_q_heads, out, T);
  if (st != DKV_OK) return st;
  if (layer < 0 || layer >= c->layers)
    return fail(DKV_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, c->layers);
  std::lock_guard<std::mutex> lk(c->mu);
  if ((st = set_device(c)) != DKV_OK) return st;
  return prefill_impl(c, layer, x, T, wq, wk, wv, hidden, n_q_heads, out, c->k_dev, c->v_dev,
                      stream);
}

dkv_status dkv_prefill_staged(dkv_cache* c, const void* x, int T, const void* wq,
                              const void* wk, const void* wv, int hidden, int n_q_heads,
                              void* out, void* k_stage, void* v_stage, void* stream) {
  dkv_status st = check_call(c, x, wq, wk, wv, hidden, n_q_heads, out, T);
  if (st != DKV_OK) return st;
  if (!k_stage || !v_stage) return fail(DKV_ERR_INVALID_ARG, "null staging buffer");
  if (c->page_tokens || c->layers != 1 || c->kv_format != DKV_KV_NATIVE)
    return fail(DKV_ERR_UNSUPPORTED, "staged prefill needs a dense one-layer 16-bit cache");
  std::lock_guard<std::mutex> lk(c->mu);
  if ((st = set_device(c)) != DKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t head_elems = (size_t)c->max_tokens * c->D;
  for (int b = 0; b < c->B; ++b)
    for (int h = 0; h < c->Hkv; ++h) {
      const size_t off = ((size_t)b * c->Hkv + h) * head_elems * 2;
      const size_t n = (size_t)c->len[b] * c->D * 2;
      if (n == 0) continue;
      cudaError_t e = cudaMemcpyAsync(static_cast<char*>(k_stage) + off,
                                      static_cast<char*>(c->k_host) + off, n,
                                      cudaMemcpyHostToDevice, s);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(static_cast<char*>(v_stage) + off,
                            static_cast<char*>(c->v_host) + off, n, cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) return cuda_fail(e, "staging cudaMemcpyAsync");
    }
  return prefill_impl(c, 0, x, T, wq, wk, wv, hidden, n_q_heads, out, k_stage, v_stage, stream);
}

dkv_status dkv_prefill_naive(dkv_cache* c, const void* x, int T, const void* wq,
                             const void* wk, const void* wv, int hidden, int n_q_heads,
                             void* out, void* stream) {
  dkv_status st = check_call(c, x, wq, wk, wv, hidden, n_q_heads, out, T);
  if (st != DKV_OK) return st;
  if (c->layers != 1 || c->kv_format != DKV_KV_NATIVE)
    return fail(DKV_ERR_UNSUPPORTED, "the naive prefill baseline needs a one-layer 16-bit cache");
  std::lock_guard<std::mutex> lk(c->mu);
  if ((st = set_device(c)) != DKV_OK) return st;
  return prefill_impl(c, 0, x, T, wq, wk, wv, hidden, n_q_heads, out, c->k_dev, c->v_dev,
                      stream, true);
}

dkv_status dkv_prefill(dkv_cache* c, const void* x, int T, const void* wq, const void* wk,
                       const void* wv, int hidden, int n_q_heads, void* out, void* stream) {
  if (valid(c) && c->layers != 1)
    return fail(DKV_ERR_INVALID_ARG, "a layered cache takes dkv_prefill_layer");
  return dkv_prefill_layer(c, 0, x, T, wq, wk, wv, hidden, n_q_heads, out, stream);
}

dkv_status dkv_cache_kernel_timing(dkv_cache* c, int enable) {
  if (!valid(c)) return fail(DKV_ERR_INVALID_ARG, "invalid cache handle");
  std::lock_guard<std::mutex> lk(c->mu);
  dkv_status st = set_device(c);
  if (st != DKV_OK) return st;
  if (enable && !c->timer.start) {
    cudaError_t e = cudaEventCreate(&c->timer.start);
    if (e == cudaSuccess) e = cudaEventCreate(&c->timer.stop);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
  } else if (!enable && c->timer.start) {
    cudaEventDestroy(c->timer.start);
    cudaEventDestroy(c->timer.stop);
    c->timer = KernelTimer();
  }
  c->timer_used = false;
  return DKV_OK;
}

dkv_status dkv_cache_last_kernel_ms(dkv_cache* c, float* ms) {
  if (!valid(c) || !ms) return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  std::lock_guard<std::mutex> lk(c->mu);
  if (!c->timer.start || !c->timer_used)
    return fail(DKV_ERR_INVALID_ARG, "kernel timing is off or nothing was recorded");
  cudaError_t e = cudaEventSynchronize(c->timer.stop);
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, c->timer.start, c->timer.stop);
  return e == cudaSuccess ? DKV_OK : cuda_fail(e, "kernel timing");
}

dkv_status dkv_sync_status(dkv_cache* c, void* stream) {
  if (!valid(c)) return fail(DKV_ERR_INVALID_ARG, "invalid cache handle");
  std::lock_guard<std::mutex> lk(c->mu);
  dkv_status st = set_device(c);
  if (st != DKV_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  DeviceStatus ds;
  e = cudaMemcpy(&ds, c->status, sizeof ds, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (ds.code != 0) {
    const int code = ds.code, site = ds.site;
    DeviceStatus z;
    memset(&z, 0, sizeof z);
    cudaMemcpy(c->status, &z, sizeof z, cudaMemcpyHostToDevice);
    return fail((dkv_status)code, "device status %d at wait site %d", code, site);
  }
  return DKV_OK;
}

dkv_status dkv_project(const void* x, const void* w, void* y, int M, int K, int N,
                       dkv_dtype dtype, void* stream) {
  if (!x || !w || !y) return fail(DKV_ERR_INVALID_ARG, "null tensor pointer");
  if (M <= 0 || K <= 0 || N <= 0 || K % 8 || N % 64)
    return fail(DKV_ERR_INVALID_ARG, "M=%d K=%d N=%d (K must be a multiple of 8, N of 64)", M,
                K, N);
  if (dtype != DKV_BF16 && dtype != DKV_FP16) return fail(DKV_ERR_INVALID_ARG, "dtype");
  cudaError_t e = launch_gemm_tc(x, w, y, M, N, K, dtype, nullptr, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "projection launch");
  }
  return DKV_OK;
}

dkv_status dkv_probe_read(const void* src, size_t bytes, void* sink, void* stream) {
  if (!src || !sink || bytes == 0 || bytes % 16) return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  cudaError_t e = launch_probe_read(src, bytes, sink, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DKV_OK : cuda_fail(e, "probe read launch");
}

dkv_status dkv_probe_write(void* dst, size_t bytes, void* stream) {
  if (!dst || bytes == 0 || bytes % 16) return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  cudaError_t e = launch_probe_write(dst, bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DKV_OK : cuda_fail(e, "probe write launch");
}

dkv_status dkv_probe_launch(int grid, int threads, int smem_bytes, void* stream) {
  if (grid < 1 || threads < 32 || threads > 1024 || threads % 32 || smem_bytes < 0 ||
      smem_bytes > 232448)
    return fail(DKV_ERR_INVALID_ARG, "invalid launch shape");
  cudaError_t e = launch_probe_empty(grid, threads, smem_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DKV_OK : cuda_fail(e, "probe launch");
}

dkv_status dkv_attend_naive(dkv_cache* c, const void* q, int n_q_heads, void* out, void* stream) {
  if (!valid(c) || !q || !out || n_q_heads <= 0 || n_q_heads % c->Hkv)
    return fail(DKV_ERR_INVALID_ARG, "invalid argument");
  if (c->page_tokens || c->layers != 1 || c->kv_format != DKV_KV_NATIVE)
    return fail(DKV_ERR_UNSUPPORTED, "naive attention needs a dense one-layer 16-bit cache");
  std::lock_guard<std::mutex> lk(c->mu);
  dkv_status st = set_device(c);
  if (st != DKV_OK) return st;
  for (int b = 0; b < c->B; ++b)
    if (c->len[b] < 1) return fail(DKV_ERR_INVALID_ARG, "sequence %d is empty", b);
  // same grid-filling rule as the fused decode: about 8 CTAs per SM
  const int units = c->B * n_q_heads;
  const int splits = std::max(1, (c->sms * 8 + units - 1) / units);
  const size_t po_b = align_up((size_t)units * splits * c->D * 4, 256);
  const size_t pl_b = align_up((size_t)units * splits * 4, 256);
  if ((st = ensure_ws(c, po_b + pl_b)) != DKV_OK) return st;
  char* w = static_cast<char*>(c->ws.base);
  cudaError_t e = launch_attend_naive(q, c->k_dev, c->v_dev, out, reinterpret_cast<float*>(w),
                                      reinterpret_cast<float*>(w + po_b), c->B, n_q_heads, c->Hkv,
                                      c->D, c->max_tokens, c->len.data(), splits, c->dtype,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "naive attention launch");
  c->last_stream = static_cast<cudaStream_t>(stream);
  return DKV_OK;
}

}  // extern "C"
