// dkv_decode_noalloc: the fused decode for callers that cannot allocate GPU
// memory.
//
// Some callers are not allowed to call cudaMalloc at all: code running inside
// an allocator or memory-pool callback, plug-ins hosted by a runtime that owns
// every device allocation, or processes that must keep a fixed memory budget
// after start-up.  For them this entry point runs the same fused decode kernel
// as dkv_decode without any allocation: its scratch (the q and fresh K/V
// workspace, the split-KV partials and the device status word) lives in one
// file-scope __device__ array of fixed size, which every GPU that loads this
// library keeps until the process exits.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>

#include "dkv_internal.cuh"

namespace dkv {
void set_last_error(dkv_status s, const char* msg);
}

namespace {

// Maximum scratch this entry point can use: 8 MiB per device.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Test hook: when set, the next calls' producers withhold their first tile's
// signal so that the consumers' bounded wait expires (process-wide).
int g_debug_withhold = 0;

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

dkv_status err(dkv_status s, const char* msg) {
  dkv::set_last_error(s, msg);
  return s;
}

// Device address of the scratch array on the current device.  The name
// g_noalloc_scratch in host code is only a host-side stand-in, so the address
// is looked up with cudaGetSymbolAddress; the lookup is repeated on every call
// (it allocates nothing), so an address never outlives the context it was
// taken in (after a cudaDeviceReset the module is loaded again elsewhere).
dkv_status scratch_address(void** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    cudaGetLastError();
    return err(DKV_ERR_CUDA, "cudaGetSymbolAddress of the no-allocation scratch failed");
  }
  *out = p;
  return DKV_OK;
}

}  // namespace

extern "C" dkv_status dkv_decode_noalloc(const void* x, const void* wq, const void* wk,
                                         const void* wv, void* k_cache, void* v_cache,
                                         const int32_t* lengths, int batch, int hidden,
                                         int n_q_heads, int n_kv_heads, int head_dim,
                                         int max_tokens, dkv_dtype dtype, void* out,
                                         void* stream) {
  using namespace dkv;
  if (!x || !wq || !wk || !wv || !k_cache || !v_cache || !lengths || !out)
    return err(DKV_ERR_INVALID_ARG, "null pointer argument");
  if (batch <= 0 || batch > kMaxBatch || n_kv_heads <= 0 || max_tokens <= 0)
    return err(DKV_ERR_INVALID_ARG, "batch, n_kv_heads or max_tokens out of range");
  if (hidden <= 0 || hidden % 16 != 0)
    return err(DKV_ERR_INVALID_ARG, "hidden must be a positive multiple of 16");
  if (n_q_heads <= 0 || n_q_heads % n_kv_heads != 0)
    return err(DKV_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
  const int G = n_q_heads / n_kv_heads;
  if (!decode_supported(dtype, head_dim, G))
    return err(DKV_ERR_UNSUPPORTED, "no decode kernel for this dtype, head_dim and group size");
  int maxS = 1;
  for (int b = 0; b < batch; ++b) {
    if (lengths[b] < 0) return err(DKV_ERR_INVALID_ARG, "negative sequence length");
    if ((long)lengths[b] + 1 > max_tokens)
      return err(DKV_ERR_CAPACITY, "length + 1 exceeds max_tokens");
    maxS = std::max(maxS, lengths[b] + 1);
  }

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return err(DKV_ERR_CUDA, "cudaGetDevice failed");
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  void* scratch = nullptr;
  dkv_status st = scratch_address(&scratch);
  if (st != DKV_OK) return st;

  // Same tile and ring as dkv_decode's default choice.
  const int D = head_dim, N = 8192 / D, stages = 4;
  int occ = 0;
  e = decode_occupancy(dtype, D, G, N, stages, batch, &occ);
  if (e != cudaSuccess || occ < 1) {
    cudaGetLastError();
    return err(DKV_ERR_CUDA, "decode kernel occupancy query failed");
  }
  const int grid = sms * occ;
  const int smem = decode_smem_bytes(dtype, D, G, N, stages, batch);

  // Scratch layout: status | q | fresh k,v | partial o | partial lse.
  const size_t st_b = align256(sizeof(DeviceStatus));
  const size_t q_b = align256((size_t)batch * n_q_heads * D * 2);
  const size_t kv_b = align256((size_t)batch * 2 * n_kv_heads * D * 2);
  auto need = [&](int s) {
    return st_b + q_b + kv_b + align256((size_t)batch * n_q_heads * s * D * 4) +
           align256((size_t)batch * n_q_heads * s * 4);
  };
  // Split count: the fewest tiles per CTA among the counts whose partials fit.
  const int nt = (maxS + N - 1) / N;
  const int bh = batch * n_kv_heads;
  int splits = 0;
  long best = -1;
  for (int s = 1; s <= std::min(nt, 1024); ++s) {
    if (need(s) > kNoAllocScratchBytes) break;
    const long units = (long)bh * s;
    const long waves = (units + grid - 1) / grid;
    const long cost = waves * ((nt + s - 1) / s) * 64 + waves;
    if (best < 0 || cost < best) { best = cost; splits = s; }
  }
  if (splits == 0) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "decode needs %zu bytes of scratch even with one split; the static scratch holds %zu",
             need(1), kNoAllocScratchBytes);
    return err(DKV_ERR_CAPACITY, msg);
  }

  char* base = static_cast<char*>(scratch);
  DecodeParams p;
  memset(&p, 0, sizeof p);
  p.x = x; p.wq = wq; p.wk = wk; p.wv = wv;
  p.k_read = k_cache; p.v_read = v_cache; p.k_host = k_cache; p.v_host = v_cache;
  p.status = reinterpret_cast<DeviceStatus*>(base);
  p.q_ws = base + st_b;
  p.kv_ws = base + st_b + q_b;
  p.part_o = reinterpret_cast<float*>(base + st_b + q_b + kv_b);
  p.part_lse = reinterpret_cast<float*>(base + st_b + q_b + kv_b +
                                        align256((size_t)batch * n_q_heads * splits * D * 4));
  p.out = out;
  p.B = batch; p.H = hidden; p.Hq = n_q_heads; p.Hkv = n_kv_heads; p.D = D;
  p.S_max = max_tokens;
  p.lay.Hkv = n_kv_heads;  // dense [B][Hkv][max_tokens][D] caches
  p.lay.S_max = max_tokens;
  p.splits = splits; p.tile_n = N; p.stages = stages;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  p.debug_withhold = g_debug_withhold;
  for (int b = 0; b < kMaxBatch; ++b) p.len[b] = b < batch ? lengths[b] : 0;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The grid-barrier counter and status word must start at zero; the array
  // keeps whatever the previous call left there.
  e = cudaMemsetAsync(p.status, 0, sizeof(DeviceStatus), s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return err(DKV_ERR_CUDA, "cudaMemsetAsync of the scratch status failed");
  }
  int launches = 0;
  e = launch_decode(p, dtype, grid, smem, s, &launches, KernelTimer());
  if (e != cudaSuccess) {
    cudaGetLastError();
    return err(DKV_ERR_CUDA, cudaGetErrorString(e));
  }
  return DKV_OK;
}

// The status of the last dkv_decode_noalloc on this device: waits for
// `stream`, reads the status word at the head of the scratch array and clears
// it.  No allocation: the word is copied into a host variable.
extern "C" dkv_status dkv_decode_noalloc_status(void* stream) {
  using namespace dkv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return err(DKV_ERR_CUDA, cudaGetErrorString(e));
  }
  DeviceStatus h;
  e = cudaMemcpyFromSymbol(&h, g_noalloc_scratch, sizeof h, 0, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return err(DKV_ERR_CUDA, "reading the no-allocation status word failed");
  }
  if (h.code == 0) return DKV_OK;
  const DeviceStatus zero = {};
  e = cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof zero, 0, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return err(DKV_ERR_CUDA, "clearing the no-allocation status word failed");
  }
  char msg[96];
  snprintf(msg, sizeof msg, "a device-side wait gave up (site %d)", h.site);
  return err(static_cast<dkv_status>(h.code), msg);
}

extern "C" dkv_status dkv_decode_noalloc_debug_withhold(int enable) {
  g_debug_withhold = enable ? 1 : 0;
  return DKV_OK;
}
