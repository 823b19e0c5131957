// Internal definitions shared by the CUDA translation units of libdkv.
// Device helpers are thin inline-PTX wrappers (mbarrier, cp.async, timers).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dkv.h"

namespace dkv {

constexpr int kMaxBatch = 64;        // sequences per call (lengths travel in the params)
constexpr uint64_t kWaitBudgetNs = 1000000000ull;  // 1 s: no legitimate wait comes close

// Device status word values (a subset of dkv_status).
constexpr int kStatusTimeout = DKV_ERR_TIMEOUT;

// Where a bounded wait gave up (recorded next to the status for diagnosis).
enum WaitSite : int {
  kSiteGridBarrier = 1,
  kSiteFull = 2,
  kSiteEmpty = 3,
};

struct DeviceStatus {
  int code;      // 0 = ok, else a dkv_status
  int site;      // WaitSite of the first timeout
  unsigned int grid_arrive;  // decode grid barrier counter (reset by the combine kernel)
  int pad;
};

// ----------------------------------------------------------------------------
// dtype traits
template <typename T> struct DT;
template <> struct DT<__nv_bfloat16> {
  static constexpr int code = DKV_BF16;
  __device__ static inline float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static inline __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
  __device__ static inline float2 to_f2(uint32_t u) {
    // two packed bf16 -> two floats (exact: a bf16 is the high half of an fp32)
    float2 r;
    r.x = __uint_as_float(u << 16);
    r.y = __uint_as_float(u & 0xFFFF0000u);
    return r;
  }
};
template <> struct DT<__half> {
  static constexpr int code = DKV_FP16;
  __device__ static inline float to_f(__half v) { return __half2float(v); }
  __device__ static inline __half from_f(float v) { return __float2half_rn(v); }
  __device__ static inline float2 to_f2(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
  }
};

// ----------------------------------------------------------------------------
// PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Programmatic dependent launch (no-ops for a kernel launched without it):
// let the next kernel in the stream launch, and wait until every earlier
// kernel has finished and its memory operations are visible.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// `count` arrivals at once (count > 0): one thread standing in for several.
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the same (never suspends the thread): for a loop that
// polls several barriers and acts on whichever completes first.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; gives up (returns
// false) once this wait has lasted kWaitBudgetNs or *abort becomes non-zero.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t deadline = global_timer_ns() + kWaitBudgetNs;
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (global_timer_ns() > deadline) return false;
  }
  return true;
}

// mbar_wait_bounded for waits that are expected to be long (a producer
// waiting for a free ring slot): between tests the thread sleeps about
// `ns` nanoseconds, leaving the issue slots to the warps that compute.
__device__ __forceinline__ bool mbar_wait_bounded_sleep(uint64_t* bar, uint32_t parity,
                                                        volatile int* abort, unsigned ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t deadline = global_timer_ns() + kWaitBudgetNs;
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (global_timer_ns() > deadline) return false;
    __nanosleep(ns);
  }
  return true;
}

// Waits, for at most the wait budget and whatever an abort flag says, for
// the phase with the given parity: after a give-up, asynchronous copies or
// MMAs already issued complete before the CTA leaves or frees what they use.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t deadline = global_timer_ns() + kWaitBudgetNs;
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() > deadline) return;
}

// 16-byte asynchronous global->shared copy; src_bytes < 16 zero-fills the rest
// (src_bytes == 0 reads nothing).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(gsrc), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The mbarrier's pending count drops by one when all of this thread's prior
// cp.async copies have landed (the barrier is initialised with one count per
// producer thread).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// A named barrier that also returns, to every participant, the OR of their
// predicates: a decision all of them take alike (e.g. to stop after an abort
// flag that another warp role may set at any moment).
__device__ __forceinline__ bool named_bar_sync_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void record_timeout(DeviceStatus* st, int site) {
  if (st && atomicCAS(&st->code, 0, kStatusTimeout) == 0) st->site = site;
}

// 16-byte chunk swizzle inside a row of `row_bytes` (>= 128): chunk c of row r
// is stored at chunk c ^ (r & 7), so 8 consecutive rows read at the same
// column hit 8 different bank groups.
__device__ __forceinline__ int swz_chunk(int r, int c) { return c ^ (r & 7); }

// ----------------------------------------------------------------------------
// Kernel parameter blocks

struct LenArray {
  int v[kMaxBatch];
};

// Where cache row `tok` of (sequence b, KV head kvh) lives, as an element
// offset from the K (or V) base.  Dense caches are [B][Hkv][S_max][D]; paged
// caches are a pool [page][Hkv][page_tokens][D] with a per-sequence page table
// (logical page i of sequence b is pool page pages[b * max_pages + i]), so a
// page holds page_tokens contiguous rows of one KV head.
struct CacheLayout {
  const int* pages;  // device [B][max_pages]; null for a dense cache
  int page_shift;    // log2(page_tokens)
  int max_pages;
  int Hkv;
  int S_max;         // dense: rows per (b, KV head)
  __device__ __forceinline__ size_t row(int b, int kvh, int tok, int D) const {
    if (!pages) return (((size_t)b * Hkv + kvh) * S_max + tok) * (size_t)D;
    const int pg = __ldg(pages + (size_t)b * max_pages + (tok >> page_shift));
    return ((((size_t)pg * Hkv + kvh) << page_shift) + (tok & ((1 << page_shift) - 1))) *
           (size_t)D;
  }
};

// What one decode launch does: the fused path, or one of the two halves of
// the separate-kernel baseline (projection + append; then attention over
// every row read from the host cache, the appended one included).
enum DecodeMode : int { kDecodeFused = 0, kDecodeProjectOnly = 1, kDecodeAttendOnly = 2 };

struct DecodeParams {
  // inputs (device)
  const void* x;    // [B, H]
  const void* wq;   // [H, Hq*D]
  const void* wk;   // [H, Hkv*D]
  const void* wv;   // [H, Hkv*D]
  // caches: rows [0, len) are read from k_read/v_read (mapped host alias or an
  // HBM staging copy); the new row is appended through k_host/v_host.
  const void* k_read;
  const void* v_read;
  void* k_host;
  void* v_host;
  // workspace (device)
  void* q_ws;      // [B, Hq*D]   dtype, q rounded
  void* kv_ws;     // [B, 2, Hkv*D] dtype, fresh k and v rounded
  float* part_o;   // [B, Hq, splits, D]
  float* part_lse; // [B, Hq, splits]  (log2 domain)
  DeviceStatus* status;
  void* out;       // [B, Hq, D]
  int B, H, Hq, Hkv, D, S_max;
  int splits;
  int tile_n;      // keys per tile
  int stages;
  float scale_log2;  // log2(e) / sqrt(D)
  int debug_withhold;  // test hook: producers never signal their first tile
  CacheLayout lay;     // rows of k_read / v_read / k_host / v_host
  int mode;            // DecodeMode
  int kv_fp8;          // caches hold 8-bit E4M3 (bf16 activations)
  // lengths: len_dev (device, [B]) when set, so that a captured graph replays
  // with the lengths of the step it runs; else the by-value copy below
  const int* len_dev;
  int len[kMaxBatch];
};

struct PrefillParams {
  const void* x;     // [B, T, H]
  const void* wk;    // [H, Hkv*D]
  const void* wv;
  const void* q;     // [B, T, Hq, D] (HBM, written by the Q projection)
  const void* k_read;
  const void* v_read;
  void* k_host;
  void* v_host;
  void* part_o;      // [nchunks, B*T*Hq, D] dtype (normalised per chunk)
  float* part_lse;   // [nchunks, B*T*Hq]  (log2 domain)
  int* part_k;       // [nchunks, B*Hkv]: partials of a chunk are stored times 2^-k
  DeviceStatus* status;
  void* out;         // [B, T, Hq, D]
  int B, T, H, Hq, Hkv, D, S_max;
  int chunk;         // keys per stationary chunk
  int nchunks;       // chunks per sequence (max over the batch)
  float scale_log2;
  CacheLayout lay;   // rows of k_read / v_read / k_host / v_host
  int naive;         // baseline: every (Q tile, chunk) pair fetches the chunk again
  int kv_fp8;        // caches hold 8-bit E4M3 (bf16 activations)
  int debug_withhold;  // test hook for the bounded-wait path
  int len[kMaxBatch];
};

// Optional event pair recorded around a call's main fused kernel.
struct KernelTimer {
  cudaEvent_t start = nullptr;
  cudaEvent_t stop = nullptr;
  void before(cudaStream_t s) const { if (start) cudaEventRecord(start, s); }
  void after(cudaStream_t s) const { if (stop) cudaEventRecord(stop, s); }
};

// Launchers (defined in the kernel translation units).
cudaError_t launch_decode(const DecodeParams& p, int dtype, int grid, int smem_bytes,
                          cudaStream_t s, int* launches, const KernelTimer& timer);
// len[b] += T for b < B (the last node of a captured decode step).
cudaError_t launch_advance_lengths(int* len, int B, int T, cudaStream_t s);
int decode_smem_bytes(int dtype, int D, int G, int tile_n, int stages, int B, bool kv_fp8 = false);
cudaError_t decode_occupancy(int dtype, int D, int G, int tile_n, int stages, int B,
                             int* blocks_per_sm, bool kv_fp8 = false);
bool decode_supported(int dtype, int D, int G);

// Tensor-core prefill (prefill_tc.cu): Q projection, fused KV-stationary
// attention with fp16 partials, combine.  Keys per stationary chunk:
bool prefill_supported(int dtype, int D, int G);
int prefill_tc_chunk_keys();
cudaError_t launch_prefill_tc(const PrefillParams& p, int dtype, const void* wq, cudaStream_t s,
                              int* launches, const KernelTimer& timer);

// Y[M,N] = X[M,K] . W[K,N] on the tensor cores (gemm_tc.cu).
cudaError_t launch_gemm_tc(const void* x, const void* w, void* y, int M, int N, int K, int dtype,
                           DeviceStatus* status, cudaStream_t s);

cudaError_t launch_probe_read(const void* src, size_t bytes, void* sink, cudaStream_t s);
cudaError_t launch_probe_write(void* dst, size_t bytes, cudaStream_t s);
cudaError_t launch_probe_empty(int grid, int threads, int smem, cudaStream_t s);
cudaError_t launch_attend_naive(const void* q, const void* k, const void* v, void* out,
                                float* part_o, float* part_lse, int B, int Hq, int Hkv, int D,
                                int S_max, const int* len, int splits, int dtype, cudaStream_t s);

}  // namespace dkv
