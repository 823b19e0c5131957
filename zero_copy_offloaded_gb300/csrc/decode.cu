// Fused decode: projection + append + split-KV attention over a host-resident
// KV cache read zero-copy, then the split-KV combine.
//
// DirectKV's decode strategy iterates over all cached (K, V) for the single
// new query ("Paper Notes: DirectKV", System Architecture, Attention Fusion
// Engine); K/V projection and attention run in one kernel with the fresh K/V
// kept on chip (Key Ideas (2)); producer warps fetch the next host tile while
// consumer warps compute on the current one (Key Ideas (3)); each host tile
// is read once and reused by every query head of its KV group (Key Ideas (1)).
//
// GB300 design: one persistent cooperative launch, one CTA per SM.
//   Phase A  every CTA projects its 32-column blocks of [Wq | Wk | Wv] for all
//            sequences (one fp32 FMA chain over H in order per output, one
//            column per thread, rounded once) and writes q and the fresh k/v
//            to a small HBM workspace.  Weight blocks and x arrive by TMA, so
//            this HBM traffic stays off the load/store path of the host
//            requests.  Meanwhile the producer warps already stream the CTA's
//            first host tiles into the shared-memory ring.
//   barrier  bounded grid-wide arrival counter (co-residency is guaranteed by
//            the cooperative launch); after its arrival each CTA copies its
//            fresh k/v rows from the workspace to the host cache (the append).
// In a captured step the kernels are programmatic dependents: the producers
// start at once, everything else waits for the earlier kernels.
//   Phase B  units (sequence b, KV head, key-range split) in a static
//            round-robin.  Producer warps copy host K/V tiles with 16-byte
//            cp.async into an m-stage ring (mbarrier hand-off), one tile in
//            flight per producer thread; consumer warps
//            compute the G heads' scores, the online softmax and P.V in fp32
//            and write one normalised partial (o, lse) per unit.
// The combine kernel merges the splits with a log-sum-exp weighting.
// The same kernel also runs the two halves of the separate-kernel baseline
// (DecodeMode): phase A alone, then phase B over rows that all come from the
// host cache, the freshly appended one included.
#include "tc_common.cuh"

#include <cuda_fp8.h>

namespace dkv {
bool make_tmap_2d_plain(CUtensorMap* map, const void* base, int dtype, uint64_t rows,
                        uint64_t cols, uint32_t box_cols, uint32_t box_rows);
namespace {

// Cache element C: the activation type T itself (2 bytes), or 8-bit E4M3
// (unscaled, saturating).  pair() turns two adjacent elements, packed in the
// low bytes of a word, into floats (element at the lower address in .x).
template <typename T, typename C>
struct KVE {
  static constexpr int EB = 2;
  __device__ static inline float2 pair(uint32_t two) { return DT<T>::to_f2(two); }
};
template <typename T>
struct KVE<T, __nv_fp8_e4m3> {
  static constexpr int EB = 1;
  __device__ static inline float2 pair(uint32_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
  }
};

// 16-byte chunk c of cache row n at chunk c ^ (n mod m), m = min(chunks per
// row, 8): rows read at the same column hit different bank groups.
template <int CPR>
__device__ __forceinline__ int swzc(int n, int c) {
  return c ^ (n & ((CPR < 8 ? CPR : 8) - 1));
}

// Cached rows of sequence b before this call's append.
__device__ __forceinline__ int seq_len(const DecodeParams& p, int b) {
  return p.len_dev ? __ldg(p.len_dev + b) : p.len[b];
}

__global__ void advance_lengths_kernel(int* len, int B, int T) {
  if (threadIdx.x < B) len[threadIdx.x] += T;
}

constexpr int kConsumerWarps = 8;
constexpr int kProducerWarps = 2;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducers = kProducerWarps * 32;
constexpr int kThreads = kConsumers + kProducers;
constexpr int kBarConsumers = 1;  // named barrier id for the consumer warps
constexpr int kProjRows = 128;    // H rows per projection chunk
constexpr int kProjBlk = 32;      // weight columns per TMA block (64-byte rows)

// Weight blocks a projection pass takes together: one thread per column and
// the batch rows split over the threads that remain, at most 8 chains a
// thread (kConsumers / 64 = 4 thread rows for two blocks, 8 for one).
__host__ __device__ inline int proj_group_max(int B) { return B <= 32 ? 2 : 1; }

constexpr int kSmemCap = 232448 - 1024;  // dynamic shared memory per CTA, with margin

// Shared-memory layout (byte offsets), all derived from the launch shape.
// The projection's staging gets as many chunk stages (4 down to 2) as fit
// beside the tile ring; a stage holds the weight blocks of one 128-row chunk
// ([block][128][32]) followed by x's matching columns for every sequence
// ([B][128]), both written by TMA.  Deeper staging keeps more HBM loads in
// flight under the in-order FMA chains.
struct DecodeSmem {
  int ring, bars, q, s, alpha, ml, red, proj, pstage, flag, total, proj_stages, pbar;
  int eb;  // bytes per cache element
  __host__ __device__ DecodeSmem(int D, int G, int N, int stages, int B, int eb_ = 2) : eb(eb_) {
    for (proj_stages = 4; proj_stages > 2; --proj_stages)
      if (layout(D, G, N, stages, B) <= kSmemCap) break;
    layout(D, G, N, stages, B);
  }
  __host__ __device__ int layout(int D, int G, int N, int stages, int B) {
    int tile_bytes = N * D * eb;
    int off = 0;
    ring = off; off += stages * 2 * tile_bytes;
    bars = off; off += 2 * stages * 8;
    q = off; off += G * (D + 4) * 4;
    s = off; off += 2 * G * N * 4;
    alpha = off; off += 2 * G * 4;
    ml = off; off += 2 * G * 4;
    red = off; off += kConsumers * 2 * 4;
    off = (off + 15) & ~15;
    off = (off + 127) & ~127;
    pstage = proj_group_max(B) * kProjRows * kProjBlk * 2 + B * kProjRows * 2;
    proj = off; off += proj_stages * pstage;
    pbar = off; off += 2 * 4 * 8;  // full[4], empty[4]
    flag = off; off += 16;
    total = off;
    return total;
  }
};

template <typename T, int D>
__device__ __forceinline__ const T* col_source(const DecodeParams& p, int col, int& which,
                                               int& local) {
  const int nq = p.Hq * D, nk = p.Hkv * D;
  if (col < nq) { which = 0; local = col; return static_cast<const T*>(p.wq); }
  if (col < nq + nk) { which = 1; local = col - nq; return static_cast<const T*>(p.wk); }
  which = 2; local = col - nq - nk; return static_cast<const T*>(p.wv);
}

// One fp32 sum rounded once to a cache element.
template <typename T, typename C>
__device__ __forceinline__ void store_one(C* dst, float a) {
  if constexpr (KVE<T, C>::EB == 1)
    *reinterpret_cast<__nv_fp8_storage_t*>(dst) = __nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3);
  else
    *dst = DT<T>::from_f(a);
}

// `rows` rows of one staged chunk into NC chains of one column: chain ci is
// batch row min(b0 + ci * bstep, B - 1) (chains past the thread's last row
// repeat a real one and are discarded).  Each step adds one exact product of
// two 16-bit floats with one fp32 rounding, rows in order.
template <typename T, int NC>
__device__ __forceinline__ void proj_rows(float (&acc)[8], const T* wcol, const T* xs, int rows,
                                          int b0, int bstep, int B) {
  const T* xr[NC];
#pragma unroll
  for (int ci = 0; ci < NC; ++ci) xr[ci] = xs + min(b0 + ci * bstep, B - 1) * kProjRows;
#pragma unroll 2
  for (int j = 0; j < rows; j += 8) {
    float w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = DT<T>::to_f(wcol[(j + k) * kProjBlk]);
#pragma unroll
    for (int ci = 0; ci < NC; ++ci) {
      const uint4 x8 = *reinterpret_cast<const uint4*>(xr[ci] + j);
      const uint32_t xw[4] = {x8.x, x8.y, x8.z, x8.w};
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        const float2 xf = DT<T>::to_f2(xw[k / 2]);
        acc[ci] = fmaf(xf.x, w[k], acc[ci]);
        acc[ci] = fmaf(xf.y, w[k + 1], acc[ci]);
      }
    }
  }
}

// Phase A: this CTA's share of the [Wq | Wk | Wv] columns for all B
// sequences.  The columns go out in 32-column blocks, block i to CTA
// i mod grid; a CTA projects up to proj_group_max(B) of its blocks per pass.
// Every output is one fp32 FMA chain over j = 0..H-1 in order, rounded once
// to T (q) or to the cache element (the fresh k/v; the host append follows
// the grid-barrier arrival, see append_rows).  Compute slot s, taken by
// consumer thread (s + 64) mod 256, owns one column and the batch rows
// b0, b0 + bstep, ...; the rotation puts the first slots on warps 2 and 3,
// whose sub-partitions no producer warp and not the issuing thread share.
// Thread 0 keeps the TMA loads of the weight blocks and of x's columns
// proj_stages chunks ahead; each warp with work in a pass releases a stage
// once it has read it, and thread 0 arrives for the warps without work,
// which skip the chunk.  Chunks are numbered across passes, so the loads run
// on over a pass boundary.
template <typename T, typename C, int D>
__device__ void project_phase(const DecodeParams& p, uint8_t* smem, const DecodeSmem& L, int ctid,
                              const CUtensorMap* mq, const CUtensorMap* mk, const CUtensorMap* mv,
                              const CUtensorMap* mx, volatile int* abort_flag) {
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.pbar);
  uint64_t* empty = full + 4;
  const int S = L.proj_stages;
  const int B = p.B, H = p.H;
  const int nblk = (p.Hq + 2 * p.Hkv) * D / kProjBlk;
  const int mine = (int)blockIdx.x < nblk ? (nblk - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  if (mine == 0) return;
  const int gmax = proj_group_max(B);
  const int nch = (H + kProjRows - 1) / kProjRows;
  const int total = ((mine + gmax - 1) / gmax) * nch;
  const int wbytes = kProjRows * kProjBlk * 2;
  const int lane = ctid % 32;
  const int slot = (ctid + 64) % kConsumers;  // compute slot of this thread

  auto issue = [&](int it) {  // thread 0: chunk it into stage it mod S
    const int ps = it / nch, c = it % nch, st = it % S;
    uint8_t* dst = smem + L.proj + st * L.pstage;
    const int kb0 = ps * gmax, nb = min(mine - kb0, gmax);
    tc::fence_proxy_async_smem();
    tc::mbar_expect_tx(&full[st], nb * wbytes + B * kProjRows * 2);
    for (int k = 0; k < nb; ++k) {
      int which, local;
      (void)col_source<T, D>(p, ((int)blockIdx.x + (kb0 + k) * (int)gridDim.x) * kProjBlk, which,
                             local);
      tc::tma_load_2d(dst + k * wbytes, which == 0 ? mq : (which == 1 ? mk : mv), local,
                      c * kProjRows, &full[st]);
    }
    tc::tma_load_2d(dst + gmax * wbytes, mx, c * kProjRows, 0, &full[st]);
  };
  int issued = 0, landed = 0;  // thread 0's count of chunks issued / known landed
  if (ctid == 0)
    for (; issued < min(S, total); ++issued) issue(issued);
  // warp 0: thread 0 refills chunk it's stage with chunk it + S once every warp
  // has read it; false (for the whole warp) after a give-up
  auto refill = [&](int it) -> bool {
    bool ok = true;
    if (ctid == 0) {
      ok = mbar_wait_bounded(&empty[it % S], (it / S) & 1, abort_flag);
      if (ok) {
        landed = max(landed, it + 1);  // chunk it was read, so it had landed
        issue(issued++);
      } else {
        if (!*abort_flag) record_timeout(p.status, kSiteEmpty);
        *abort_flag = 1;
      }
    }
    return __shfl_sync(0xffffffffu, ok, 0);
  };

  float acc[8];
  for (int it = 0; it < total; ++it) {
    const int ps = it / nch, c = it % nch, st = it % S;
    const uint32_t ph = (it / S) & 1;
    const int kb0 = ps * gmax, nb = min(mine - kb0, gmax);
    const int ncc = nb * kProjBlk;                 // columns of this pass
    const int bstep = kConsumers / ncc;            // thread rows
    const int col = slot % ncc, b0 = slot / ncc;   // warp-uniform b0
    const bool active = b0 < bstep && b0 < B;
    const int nc = active ? (B - b0 + bstep - 1) / bstep : 0;  // chains of this thread
    const int ncmax = (B + bstep - 1) / bstep;                 // ... of the busiest thread
    const int nslots = ncc * min(bstep, B);        // active slots: 0 .. nslots-1
    const int nwarps = (nslots + 31) / 32;         // warps with work in this pass
    const bool wact = slot / 32 < nwarps;          // this warp has work
    if (c == 0) {
#pragma unroll
      for (int ci = 0; ci < 8; ++ci) acc[ci] = 0.f;
    }
    if (ctid == 0 && nwarps < kConsumerWarps)
      mbar_arrive_cnt(&empty[st], kConsumerWarps - nwarps);  // for the warps without work
    if (!wact) {
      if (ctid < 32 && it + S < total && !refill(it)) break;  // warp 0 still refills
      continue;
    }
    // (warp-uniform decisions: the lanes of a warp leave the loop together)
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[st], ph, abort_flag))) {
      if (lane == 0) {
        if (!*abort_flag) record_timeout(p.status, kSiteFull);
        *abort_flag = 1;
      }
      break;
    }
    landed = it + 1;
    if (active) {
      const uint8_t* stage = smem + L.proj + st * L.pstage;
      const T* wcol = reinterpret_cast<const T*>(stage + (col / kProjBlk) * wbytes) + col % kProjBlk;
      const T* xs = reinterpret_cast<const T*>(stage + gmax * wbytes);
      const int rows = min(kProjRows, H - c * kProjRows);  // a multiple of 16
      if (ncmax <= 1) proj_rows<T, 1>(acc, wcol, xs, rows, b0, bstep, B);
      else if (ncmax <= 2) proj_rows<T, 2>(acc, wcol, xs, rows, b0, bstep, B);
      else if (ncmax <= 4) proj_rows<T, 4>(acc, wcol, xs, rows, b0, bstep, B);
      else proj_rows<T, 8>(acc, wcol, xs, rows, b0, bstep, B);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    if (c == nch - 1 && active) {
      int which, local;
      (void)col_source<T, D>(p, ((int)blockIdx.x + (kb0 + col / kProjBlk) * (int)gridDim.x) *
                                        kProjBlk + col % kProjBlk,
                             which, local);
#pragma unroll
      for (int ci = 0; ci < 8; ++ci) {
        if (ci >= nc) break;
        const int b = b0 + ci * bstep;
        if (which == 0)
          static_cast<T*>(p.q_ws)[(size_t)b * p.Hq * D + local] = DT<T>::from_f(acc[ci]);
        else
          store_one<T, C>(static_cast<C*>(p.kv_ws) + ((size_t)b * 2 + (which - 1)) * p.Hkv * D +
                              local,
                          acc[ci]);
      }
    }
    if (ctid < 32 && it + S < total && !refill(it)) break;
  }
  // after a give-up, the loads already issued land before the CTA moves on
  // (bounded).  Chunks [landed, issued) are at most S consecutive ones, one per
  // stage, each the stage's latest use, so each parity names its own phase.
  if (ctid == 0 && *abort_flag)
    for (int i = landed; i < issued; ++i) mbar_wait_drain(&full[i % S], (i / S) & 1);
}

// The append: the fresh k/v of this CTA's projection blocks, copied from the
// workspace to the new row of the host cache, 16 bytes at a time (a block's
// 32 columns are contiguous in both).  The fused kernel runs it after its
// grid-barrier arrival, so the fence before that arrival does not wait for
// writes across the link.
template <typename T, typename C, int D>
__device__ void append_rows(const DecodeParams& p, int ctid) {
  constexpr int CB = kProjBlk * (int)sizeof(C) / 16;  // 16-byte pieces per block row
  const int nq = p.Hq * D, nkv = p.Hkv * D;
  const int nblk = (p.Hq + 2 * p.Hkv) * D / kProjBlk;
  const int mine = (int)blockIdx.x < nblk ? (nblk - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  for (int i = ctid; i < mine * p.B * CB; i += kConsumers) {
    const int piece = i % CB, b = (i / CB) % p.B, k = i / (CB * p.B);
    const int col0 = ((int)blockIdx.x + k * (int)gridDim.x) * kProjBlk;
    if (col0 < nq) continue;  // a q block
    const int which = col0 < nq + nkv ? 0 : 1;  // k or v
    const int local = col0 - nq - which * nkv;
    const C* src = static_cast<const C*>(p.kv_ws) + ((size_t)b * 2 + which) * nkv + local;
    C* dst = static_cast<C*>(which == 0 ? p.k_host : p.v_host) +
             p.lay.row(b, local / D, seq_len(p, b), D) + local % D;
    reinterpret_cast<uint4*>(dst)[piece] = __ldcg(reinterpret_cast<const uint4*>(src) + piece);
  }
}

struct UnitRange {
  int b, kvh, split, t_lo, t_hi, S;
};

__device__ __forceinline__ UnitRange unit_range(const DecodeParams& p, int u) {
  UnitRange r;
  r.split = u % p.splits;
  const int bh = u / p.splits;
  r.kvh = bh % p.Hkv;
  r.b = bh / p.Hkv;
  r.S = seq_len(p, r.b) + 1;  // keys after the append
  const int nt = (r.S + p.tile_n - 1) / p.tile_n;
  r.t_lo = (int)((long long)r.split * nt / p.splits);
  r.t_hi = (int)((long long)(r.split + 1) * nt / p.splits);
  return r;
}

template <typename T, typename C, int D, int G>
__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(
    const __grid_constant__ CUtensorMap map_wq, const __grid_constant__ CUtensorMap map_wk,
    const __grid_constant__ CUtensorMap map_wv, const __grid_constant__ CUtensorMap map_x,
    const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int EB = KVE<T, C>::EB;
  constexpr int RB = D * EB;   // bytes per cache row
  constexpr int EPC = 16 / EB; // elements per 16-byte chunk
  const int N = p.tile_n, stages = p.stages;
  const DecodeSmem L(D, G, N, stages, p.B, EB);
  const int tid = threadIdx.x;
  const int tile_bytes = N * RB;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.flag);

  griddep_launch_dependents();  // (no-op unless launched as a programmatic primary)
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], kProducers);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    uint64_t* pb = reinterpret_cast<uint64_t*>(smem + L.pbar);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&pb[s], 1);                    // projection stage s loaded
      mbar_init(&pb[4 + s], kConsumerWarps);  // ... and read by every consumer warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int nunits = p.B * p.Hkv * p.splits;
  constexpr int CPR = RB / 16;  // 16-byte chunks per row

  if (tid >= kConsumers) {
    // ------------------------------------------------------------ producer
    if (p.mode == kDecodeProjectOnly) return;
    const int ptid = tid - kConsumers;
    int it = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      const UnitRange r = unit_range(p, u);
      const C* kg = static_cast<const C*>(p.k_read);
      const C* vg = static_cast<const C*>(p.v_read);
      // rows read from the host: the cached ones (the fused path takes the new
      // row from HBM), or every row when the projection ran as its own launch
      const int cached = seq_len(p, r.b) + (p.mode == kDecodeAttendOnly ? 1 : 0);
      for (int t = r.t_lo; t < r.t_hi; ++t, ++it) {
        const int stage = it % stages;
        const uint32_t par = ((it / stages) & 1) ^ 1;
        if (!mbar_wait_bounded_sleep(&empty[stage], par, abort_flag, 256)) {
          if (!*abort_flag) record_timeout(p.status, kSiteEmpty);
          *abort_flag = 1;
          cp_async_wait_all();
          return;
        }
        uint8_t* kt = smem + L.ring + stage * 2 * tile_bytes;
        uint8_t* vt = kt + tile_bytes;
        const int key0 = t * N;
        const int nrows = max(0, min(N, cached - key0));
        for (int i = ptid; i < nrows * CPR; i += kProducers) {
          const int row = i / CPR, c = i % CPR;
          const int dst = row * RB + swzc<CPR>(row, c) * 16;
          const size_t src = p.lay.row(r.b, r.kvh, key0 + row, D) + c * EPC;
          cp_async16(kt + dst, kg + src, 16);
          cp_async16(vt + dst, vg + src, 16);
        }
        // (the test hook withholds the first tile's signal: the consumers'
        // bounded wait then expires and reports a timeout)
        if (!(p.debug_withhold && it == 0)) cp_async_arrive_noinc(&full[stage]);
        // One tile in flight per producer thread (32 KB per SM keeps the link
        // busy): thousands of outstanding host requests would otherwise hold
        // up the projection's weight loads on the same load/store path.
        cp_async_commit();
        cp_async_wait_group<0>();
      }
    }
    cp_async_wait_all();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = tid;
  const int warp = ctid / 32, lane = ctid % 32;

  // Under a programmatic dependent launch the producers stream the cached rows
  // (written by earlier steps) at once; x, the workspace and the barrier
  // counter belong to earlier kernels until they have finished.
  griddep_wait();
  // Phase A: this CTA's projection blocks.
  if (p.mode != kDecodeAttendOnly)
    project_phase<T, C, D>(p, smem, L, ctid, &map_wq, &map_wk, &map_wv, &map_x, abort_flag);
  if (p.mode == kDecodeProjectOnly) {  // (the producers returned at once)
    named_bar_sync(kBarConsumers, kConsumers);
    if (!*abort_flag) append_rows<T, C, D>(p, ctid);
    return;
  }
  if (p.mode == kDecodeFused) {
    // Grid barrier: every CTA's q and fresh k/v are in the workspace.  (The
    // attention-only launch follows the projection launch on the stream.)
    named_bar_sync(kBarConsumers, kConsumers);
    if (ctid == 0) {
      __threadfence();
      atomicAdd(&p.status->grid_arrive, 1u);
    }
    if (!*abort_flag) append_rows<T, C, D>(p, ctid);
    if (ctid == 0) {
      const uint64_t deadline = global_timer_ns() + kWaitBudgetNs;
      while (ld_acquire_gpu(&p.status->grid_arrive) < gridDim.x) {
        if (global_timer_ns() > deadline) {
          record_timeout(p.status, kSiteGridBarrier);
          *abort_flag = 1;
          break;
        }
      }
    }
    // one decision for all consumers: a producer may raise the flag between
    // two of them reading it, and a consumer that went on alone would wait at
    // the next named barrier for warps that had left
    if (named_bar_sync_or(kBarConsumers, kConsumers, *abort_flag != 0)) return;
  }

  float* q_s = reinterpret_cast<float*>(smem + L.q);     // [G][D+4]
  float* s_s = reinterpret_cast<float*>(smem + L.s);     // [2][G][N]
  float* alpha_s = reinterpret_cast<float*>(smem + L.alpha);  // [2][G]
  float* m_s = reinterpret_cast<float*>(smem + L.ml);    // [G]
  float* l_s = m_s + G;                                  // [G]
  float* red_s = reinterpret_cast<float*>(smem + L.red); // [kConsumers][2]

  // score mapping
  const int NS = N * G;
  const int TPS = NS >= kConsumers ? 1 : kConsumers / NS;   // threads per score
  const int SPT = NS > kConsumers ? NS / kConsumers : 1;    // scores per thread
  const int DPT = D / TPS;                                  // dims per thread
  // P.V mapping
  constexpr int NP = G * D / 2;                                   // output pairs
  constexpr int KG = NP >= kConsumers ? 1 : kConsumers / NP;      // key groups
  constexpr int PPT = NP > kConsumers ? NP / kConsumers : 1;      // pairs per thread
  constexpr int TPG = kConsumers / KG;                            // threads per key group
  const int kgi = ctid / TPG;

  int it = 0;
  for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
    const UnitRange r = unit_range(p, u);
    // q of the G heads of this KV group (bf16/fp16 values, held as fp32)
    for (int i = ctid; i < G * D; i += kConsumers) {
      const int g = i / D, d = i % D;
      const T* qg = static_cast<const T*>(p.q_ws) + (size_t)r.b * p.Hq * D + (r.kvh * G + g) * D + d;
      q_s[g * (D + 4) + d] = DT<T>::to_f(__ldcg(qg));
    }
    float acc[PPT][2];
#pragma unroll
    for (int pp = 0; pp < PPT; ++pp) acc[pp][0] = acc[pp][1] = 0.f;

    for (int t = r.t_lo; t < r.t_hi; ++t, ++it) {
      const int stage = it % stages;
      const uint32_t par = (it / stages) & 1;
      const int buf = it & 1;
      const int key0 = t * N;
      const int nvalid = min(N, r.S - key0);
      uint8_t* kt = smem + L.ring + stage * 2 * tile_bytes;
      uint8_t* vt = kt + tile_bytes;
      if (ctid == 0) {
        if (!mbar_wait_bounded(&full[stage], par, abort_flag)) {
          if (!*abort_flag) record_timeout(p.status, kSiteFull);
          *abort_flag = 1;
        }
      }
      // the new token's row (if in this tile) comes from the HBM workspace
      const int rnew = seq_len(p, r.b) - key0;
      if (p.mode == kDecodeFused && rnew >= 0 && rnew < N && ctid < 2 * CPR) {
        const int which = ctid / CPR, c = ctid % CPR;
        const C* src = static_cast<const C*>(p.kv_ws) +
                       ((size_t)r.b * 2 + which) * p.Hkv * D + r.kvh * D + c * EPC;
        uint8_t* dst = (which ? vt : kt) + rnew * RB + swzc<CPR>(rnew, c) * 16;
        *reinterpret_cast<uint4*>(dst) = __ldcg(reinterpret_cast<const uint4*>(src));
      }
      if (named_bar_sync_or(kBarConsumers, kConsumers, *abort_flag != 0)) return;

      // scores s[g][n] = (q_g . k_n) * log2(e)/sqrt(D)
      float* sb = s_s + buf * G * N;
      for (int si = 0; si < SPT; ++si) {
        const int sc = ctid / TPS + si * (kConsumers / TPS);
        const int n = sc / G, g = sc % G;
        const int part = ctid % TPS;
        float dot = 0.f;
        if (n < nvalid) {
          const float* qrow = q_s + g * (D + 4) + part * DPT;
          const uint8_t* krow = kt + n * RB;
#pragma unroll 4
          for (int c8 = 0; c8 < DPT / EPC; ++c8) {
            const int c = part * (DPT / EPC) + c8;
            const uint4 kv = *reinterpret_cast<const uint4*>(krow + swzc<CPR>(n, c) * 16);
            const uint32_t w4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int e = 0; e < EPC / 2; ++e) {
              // pair e of the chunk: word e (16-bit elements) or half-word e (8-bit)
              const uint32_t two = EB == 2 ? w4[e] : (w4[e / 2] >> (16 * (e % 2)));
              const float2 k = KVE<T, C>::pair(two);
              const float2 q = *reinterpret_cast<const float2*>(qrow + c8 * EPC + 2 * e);
              dot = fmaf(q.x, k.x, dot);
              dot = fmaf(q.y, k.y, dot);
            }
          }
        }
        for (int off = TPS / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        if (part == 0 && n < N) sb[g * N + n] = n < nvalid ? dot * p.scale_log2 : -INFINITY;
      }
      named_bar_sync(kBarConsumers, kConsumers);

      // online softmax, one warp per head
      const bool first = (t == r.t_lo);
      if (warp < G) {
        const int g = warp;
        float mx = -INFINITY;
        for (int n = lane; n < N; n += 32) mx = fmaxf(mx, sb[g * N + n]);
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_old = first ? -INFINITY : m_s[g];
        const float l_old = first ? 0.f : l_s[g];
        const float m_new = fmaxf(m_old, mx);
        float sum = 0.f;
        for (int n = lane; n < N; n += 32) {
          const float e = exp2f(sb[g * N + n] - m_new);
          sb[g * N + n] = e;
          sum += e;
        }
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane == 0) {
          const float a = exp2f(m_old - m_new);
          alpha_s[buf * G + g] = a;
          m_s[g] = m_new;
          l_s[g] = a * l_old + sum;
        }
      }
      named_bar_sync(kBarConsumers, kConsumers);

      // O = alpha * O + P . V
#pragma unroll
      for (int pp = 0; pp < PPT; ++pp) {
        const int pi = ctid % TPG + pp * TPG;
        const int g = pi / (D / 2), dp = pi % (D / 2);
        const float a = alpha_s[buf * G + g];
        float o0 = acc[pp][0] * a, o1 = acc[pp][1] * a;
        const float* prow = sb + g * N;
        const int c = dp / (EPC / 2), within = (dp % (EPC / 2)) * 2 * EB;
        for (int n = kgi; n < nvalid; n += KG) {
          const float pw = prow[n];
          const uint8_t* vp = vt + n * RB + swzc<CPR>(n, c) * 16 + within;
          const uint32_t v2 = EB == 2 ? *reinterpret_cast<const uint32_t*>(vp)
                                      : (uint32_t)*reinterpret_cast<const uint16_t*>(vp);
          const float2 v = KVE<T, C>::pair(v2);
          o0 = fmaf(pw, v.x, o0);
          o1 = fmaf(pw, v.y, o1);
        }
        acc[pp][0] = o0;
        acc[pp][1] = o1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }

    // unit end: fold the key groups, normalise, write the partial
    if (KG > 1) {
      red_s[ctid * 2] = acc[0][0];
      red_s[ctid * 2 + 1] = acc[0][1];
    }
    named_bar_sync(kBarConsumers, kConsumers);
    if (kgi == 0) {
#pragma unroll
      for (int pp = 0; pp < PPT; ++pp) {
        const int pi = ctid % TPG + pp * TPG;
        const int g = pi / (D / 2), dp = pi % (D / 2);
        float o0 = acc[pp][0], o1 = acc[pp][1];
        if (KG > 1) {
          for (int k = 1; k < KG; ++k) {
            o0 += red_s[(ctid + k * TPG) * 2];
            o1 += red_s[(ctid + k * TPG) * 2 + 1];
          }
        }
        const int h = r.kvh * G + g;
        const size_t slot = ((size_t)r.b * p.Hq + h) * p.splits + r.split;
        const bool empty_unit = r.t_hi <= r.t_lo;
        const float l = empty_unit ? 1.f : l_s[g];
        float2 o = make_float2(empty_unit ? 0.f : o0 / l, empty_unit ? 0.f : o1 / l);
        *reinterpret_cast<float2*>(p.part_o + slot * D + dp * 2) = o;
        if (dp == 0) p.part_lse[slot] = empty_unit ? -INFINITY : m_s[g] + log2f(l);
      }
    }
    named_bar_sync(kBarConsumers, kConsumers);
  }
}

// Split-KV combine: o = sum_i 2^(lse_i - M) o_i / sum_i 2^(lse_i - M).
// If a device-side wait of the fused kernel gave up (the status word holds an
// error), some partials were never written: the outputs are NaN instead of a
// merge of stale scratch.
template <typename T>
__global__ void decode_combine_kernel(const float* __restrict__ part_o,
                                      const float* __restrict__ part_lse, T* __restrict__ out,
                                      int splits, int D, DeviceStatus* status) {
  // (launched as a programmatic dependent inside a captured step: the next
  // kernel may launch now; this one reads nothing before the fused kernel ends)
  griddep_launch_dependents();
  griddep_wait();
  const int bh = blockIdx.x;
  if (*(volatile int*)&status->code != 0) {
    for (int d = threadIdx.x; d < D; d += blockDim.x) out[(size_t)bh * D + d] = DT<T>::from_f(NAN);
    if (blockIdx.x == 0 && threadIdx.x == 0) status->grid_arrive = 0u;
    return;
  }
  const float* lse = part_lse + (size_t)bh * splits;
  float M = -INFINITY;
  for (int i = 0; i < splits; ++i) M = fmaxf(M, lse[i]);
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float num = 0.f, den = 0.f;
    for (int i = 0; i < splits; ++i) {
      const float w = exp2f(lse[i] - M);
      num = fmaf(w, part_o[((size_t)bh * splits + i) * D + d], num);
      den += w;
    }
    out[(size_t)bh * D + d] = DT<T>::from_f(num / den);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) status->grid_arrive = 0u;
}

template <typename T, typename C, int D, int G>
cudaError_t launch_decode_t(const DecodeParams& p, int grid, int smem, cudaStream_t s,
                            const KernelTimer& timer) {
  auto kern = decode_fused_kernel<T, C, D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // tensor maps for phase A's TMA loads: 32-column x 128-row weight blocks
  // and x's 128 columns of every sequence (x is [B, H])
  CUtensorMap mq, mk, mv, mx;
  memset(&mq, 0, sizeof mq);
  memset(&mk, 0, sizeof mk);
  memset(&mv, 0, sizeof mv);
  memset(&mx, 0, sizeof mx);
  const int dt = std::is_same<T, __nv_bfloat16>::value ? DKV_BF16 : DKV_FP16;
  if (p.mode != kDecodeAttendOnly &&
      (!make_tmap_2d_plain(&mq, p.wq, dt, p.H, (uint64_t)p.Hq * D, kProjBlk, kProjRows) ||
       !make_tmap_2d_plain(&mk, p.wk, dt, p.H, (uint64_t)p.Hkv * D, kProjBlk, kProjRows) ||
       !make_tmap_2d_plain(&mv, p.wv, dt, p.H, (uint64_t)p.Hkv * D, kProjBlk, kProjRows) ||
       !make_tmap_2d_plain(&mx, p.x, dt, p.B, p.H, kProjRows, p.B)))
    return cudaErrorInvalidValue;
  timer.before(s);
  if (p.len_dev) {
    // the form a stream capture records as a cooperative graph node
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    // Programmatic dependent launch: the next layer's kernel may start on the
    // SMs this one leaves and stream its host tiles; whatever it reads or
    // writes that earlier kernels touch waits for them (griddepcontrol.wait).
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mx, p);
  } else {
    void* args[] = {&mq, &mk, &mv, &mx, const_cast<DecodeParams*>(&p)};
    e = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kThreads), args,
                                    (size_t)smem, s);
  }
  if (e != cudaSuccess) return e;
  timer.after(s);
  if (p.mode == kDecodeProjectOnly) return cudaSuccess;
  if (p.len_dev) {  // captured: a programmatic dependent of the fused kernel
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B * p.Hq);
    cfg.blockDim = dim3(D);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<T>, (const float*)p.part_o,
                              (const float*)p.part_lse, static_cast<T*>(p.out), p.splits, D,
                              p.status);
  }
  decode_combine_kernel<T><<<p.B * p.Hq, D, 0, s>>>(p.part_o, p.part_lse,
                                                    static_cast<T*>(p.out), p.splits, D,
                                                    p.status);
  return cudaGetLastError();
}

template <typename T, typename C, int D, int G>
cudaError_t occupancy_t(int smem, int* blocks) {
  auto kern = decode_fused_kernel<T, C, D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, kern, kThreads, smem);
}

// Kernel repository: <activation type, cache element, head_dim, group size>
// instantiations; `dtype` is the activation dtype, kv_fp8 selects E4M3 caches
// (bf16 activations only).
template <typename F>
cudaError_t dispatch(int dtype, bool kv_fp8, int D, int G, F&& f) {
#define DKV_CASE(TT, DD, GG) \
  if (D == DD && G == GG) return f.template operator()<TT, TT, DD, GG>();
#define DKV_CASE8(DD, GG) \
  if (D == DD && G == GG) return f.template operator()<__nv_bfloat16, __nv_fp8_e4m3, DD, GG>();
  if (kv_fp8) {
    if (dtype != DKV_BF16) return cudaErrorInvalidValue;
    DKV_CASE8(64, 1) DKV_CASE8(64, 2) DKV_CASE8(64, 4) DKV_CASE8(64, 8)
    DKV_CASE8(128, 1) DKV_CASE8(128, 2) DKV_CASE8(128, 4) DKV_CASE8(128, 8)
  } else if (dtype == DKV_BF16) {
    DKV_CASE(__nv_bfloat16, 64, 1) DKV_CASE(__nv_bfloat16, 64, 2) DKV_CASE(__nv_bfloat16, 64, 4)
    DKV_CASE(__nv_bfloat16, 64, 8) DKV_CASE(__nv_bfloat16, 128, 1) DKV_CASE(__nv_bfloat16, 128, 2)
    DKV_CASE(__nv_bfloat16, 128, 4) DKV_CASE(__nv_bfloat16, 128, 8)
  } else {
    DKV_CASE(__half, 64, 1) DKV_CASE(__half, 64, 2) DKV_CASE(__half, 64, 4)
    DKV_CASE(__half, 64, 8) DKV_CASE(__half, 128, 1) DKV_CASE(__half, 128, 2)
    DKV_CASE(__half, 128, 4) DKV_CASE(__half, 128, 8)
  }
#undef DKV_CASE
#undef DKV_CASE8
  return cudaErrorInvalidValue;
}

}  // namespace

bool decode_supported(int dtype, int D, int G) {
  return (dtype == DKV_BF16 || dtype == DKV_FP16) && (D == 64 || D == 128) &&
         (G == 1 || G == 2 || G == 4 || G == 8);
}

cudaError_t launch_advance_lengths(int* len, int B, int T, cudaStream_t s) {
  advance_lengths_kernel<<<1, 64, 0, s>>>(len, B, T);
  return cudaGetLastError();
}

int decode_smem_bytes(int dtype, int D, int G, int tile_n, int stages, int B, bool kv_fp8) {
  (void)dtype;
  return DecodeSmem(D, G, tile_n, stages, B, kv_fp8 ? 1 : 2).total;
}

struct LaunchDecodeF {
  const DecodeParams* p; int grid; int smem; cudaStream_t s; const KernelTimer* timer;
  template <typename T, typename C, int D, int G> cudaError_t operator()() {
    return launch_decode_t<T, C, D, G>(*p, grid, smem, s, *timer);
  }
};
struct OccF {
  int smem; int* blocks;
  template <typename T, typename C, int D, int G> cudaError_t operator()() {
    return occupancy_t<T, C, D, G>(smem, blocks);
  }
};

cudaError_t launch_decode(const DecodeParams& p, int dtype, int grid, int smem_bytes,
                          cudaStream_t s, int* launches, const KernelTimer& timer) {
  LaunchDecodeF f{&p, grid, smem_bytes, s, &timer};
  cudaError_t e = dispatch(dtype, p.kv_fp8 != 0, p.D, p.Hq / p.Hkv, f);
  if (e == cudaSuccess && launches) *launches += p.mode == kDecodeProjectOnly ? 1 : 2;
  return e;
}

cudaError_t decode_occupancy(int dtype, int D, int G, int tile_n, int stages, int B,
                             int* blocks_per_sm, bool kv_fp8) {
  OccF f{decode_smem_bytes(dtype, D, G, tile_n, stages, B, kv_fp8), blocks_per_sm};
  return dispatch(dtype, kv_fp8, D, G, f);
}

}  // namespace dkv
