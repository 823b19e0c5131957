// Fused KV-stationary prefill on the 5th-generation tensor cores.
//
// DirectKV's prefill holds each (K, V) tile fetched from host memory
// stationary and iterates over the HBM-resident Q ("Paper Notes: DirectKV",
// System Architecture, Attention Fusion Engine; Key Ideas (1)); the K/V
// projection of new tokens is fused so the fresh K/V are produced on chip and
// consumed there (Key Ideas (2)); warps specialise into loading, computing and
// storing roles (Key Ideas (3)).
//
// One CTA = one unit (sequence b, KV head, chunk of C = 256 keys).
//   1. The chunk's K and V land in shared memory (128-byte swizzled rows):
//      cached rows with 16-byte cp.async from the mapped host cache (each host
//      byte crosses the link once), new rows from a tcgen05 GEMM
//      [x rows] . [Wk | Wv] (TMA-fed, 128 rows per pass, each pass
//      accumulating in its own TMEM columns) whose epilogue rounds them,
//      writes them into the stationary tile and appends them to the host
//      cache in whole 128-byte lines.
//   2. Every Q tile of the KV group that can see the chunk (128 rows = 128/G
//      tokens x G heads, TMA from HBM) runs S = Q.K^T (tcgen05, N = 256, TMEM),
//      a complete softmax over the chunk (it is stationary, so there is no
//      running rescale), O = P.V (tcgen05 with P as the TMEM operand, fp16),
//      and its normalised O (staged in shared memory, TMA store) and base-2
//      log-sum-exp are written as the chunk's partial.  Two Q tiles are in
//      flight, each in its own TMEM region, so the tensor cores compute one
//      tile's S or O while the other tile's softmax or epilogue runs.
// A combine kernel merges the chunks' partials per query row.
//
// Warp roles (320 threads): warp 0 loads (TMA / cp.async), warp 1 allocates
// TMEM and issues every MMA from one thread, warps 2-9 are two softmax /
// epilogue groups of four (one warp per TMEM lane quarter, one row per
// thread): group 0 takes the even Q tiles, group 1 the odd ones.  Every wait
// is bounded.
#include <cuda_fp8.h>

#include <type_traits>

#include "tc_common.cuh"

namespace dkv {

bool make_tmap_2d(CUtensorMap* map, const void* base, int dtype, uint64_t rows, uint64_t cols,
                  uint32_t box_cols, uint32_t box_rows);
bool make_tmap_q(CUtensorMap* map, const void* q, int dtype, int D, int Hq, uint64_t tokens,
                 int G, int TQ);
bool make_tmap_partial(CUtensorMap* map, void* base, int D, uint64_t rows, uint64_t blocks);

namespace {

constexpr int kC = 256;        // keys per stationary chunk
constexpr int kBQ = 128;       // rows per Q tile
constexpr int kThreads = 320;  // 10 warps
constexpr int kRegKV = kC * 128;   // one 256-row x 128-byte swizzled region (K or V)
constexpr int kRegQ = kBQ * 128;   // one 128-row x 128-byte swizzled region
// TMEM: two regions of 256 columns, one per Q tile in flight (tile i uses
// region i & 1).  A region holds S (256 fp32 columns); the softmax then writes
// P (256 fp16 keys, two per column) over columns 0..127 of the consumed
// scores, and P.V accumulates O (D fp32 columns) in columns 128..128+D-1.
constexpr uint32_t kTmRegion = 256;
constexpr uint32_t kTmP = 0;
constexpr uint32_t kTmO = 128;

template <int D>
struct TcCfg {
  // projection staging stages: four where shared memory has room (D = 64,
  // 192 KB), two at D = 128 (they fill the Q buffers and the output staging)
  static constexpr int SP = D == 64 ? 4 : 2;
  static constexpr int DR = D / 64;                    // 128-byte regions per row
  static constexpr int kKV = DR * kRegKV;              // one of K or V
  static constexpr int kQ = DR * kRegQ;                // one Q tile
  static constexpr int kO = DR * kRegQ;                // output staging (128 rows)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKV;
  static constexpr int kOffQ = kOffV + kKV;            // two Q buffers
  static constexpr int kOffO = kOffQ + 2 * kQ;
  // projection staging (aliases the Q buffers, the output staging and what
  // follows): x block [128 x 64] and W block [64 x 2D], SP stages
  static constexpr int kProjA = kBQ * 64 * 2;          // 16 KB
  static constexpr int kProjB = 64 * 2 * D * 2;        // 16 / 32 KB
  static constexpr int kProjStage = kProjA + kProjB;
  static constexpr int kEnd = (kOffO + kO) > (kOffQ + SP * kProjStage) ? (kOffO + kO)
                                                                        : (kOffQ + SP * kProjStage);
  static constexpr int kOffBar = kEnd;
};

constexpr int kSmemLimit = 232448;  // 227 KB of dynamic shared memory per CTA

template <int D>
constexpr int smem_request() {
  // tiles + barrier block + up to 1 KB to align the tiles to 1024 bytes, capped
  // at the per-CTA limit (the kernel checks the padding it actually needs)
  return (TcCfg<D>::kEnd + 4096 + 1024) < kSmemLimit ? (TcCfg<D>::kEnd + 4096 + 1024)
                                                      : kSmemLimit;
}

struct Bars {
  uint64_t q_full[2], q_empty[2], kv_host, kv_ready, pr_full[4], pr_empty[4];
  // one phase each: projection pass p's MMAs have completed (pr_done[p]);
  // every pass's MMAs have completed (pr_all: the loader's signal that the
  // staging it aliases with the Q buffers is free)
  uint64_t pr_done[2], pr_all;
  // one phase each: the four warps of epilogue half h have written pass p's
  // rows into the stationary tile (they then append those rows from it)
  uint64_t ap_sync[2][2];
  // per TMEM region: S computed, P written (4 warps), O computed, O read out
  // (4 warps: the region may take the next tile's S)
  uint64_t s_full[2], p_full[2], o_full[2], r_free[2];
  // per lane quarter: the output staging rows were read by the TMA store of
  // the previous tile (the other group's), one arrival per tile
  uint64_t st_free[4];
  uint64_t vsync;     // rendezvous of the four warps converting V
  uint64_t mma_drain; // after a give-up: every MMA the issuing thread started has completed
  uint32_t tmem_base;
  volatile int abort;
  float vmax[4];
};

struct TcArgs {
  const void* k_read;
  const void* v_read;
  void* k_host;
  void* v_host;
  void* part_o;     // [nchunks, B, Hkv, T, G, D] fp16, normalised, times 2^-k of the chunk
  float* part_lse;  // [nchunks, B, Hkv, T, G]
  int* part_k;      // [nchunks, B*Hkv]
  DeviceStatus* status;
  int B, T, H, Hq, Hkv, nchunks;
  // Q tiles per CTA.  The fused prefill gives each CTA every Q tile of its
  // chunk (tile_groups = 1); the naive baseline gives each CTA one group of
  // tiles_per_group tiles, so the chunk is fetched once per group.
  int tile_groups, tiles_per_group;
  int new_first;  // fused prefill: launch the units holding new tokens first
  int nsplit;     // with new_first: the last nsplit prefix units run as two
                  // CTAs each, one per half of the chunk's Q tiles
  int debug_withhold;  // test hook: the loader never signals the chunk's host rows
  CacheLayout lay;  // rows of the caches (dense or paged)
  float scale_log2;
  int len[kMaxBatch];
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* bars,
                                              DeviceStatus* st, int site) {
  if (mbar_wait_bounded(bar, parity, &bars->abort)) return true;
  if (!bars->abort) record_timeout(st, site);
  bars->abort = 1;
  return false;
}

// Warp-uniform bounded wait (tcgen05.ld / st after it need the whole warp).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, Bars* bars,
                                          DeviceStatus* st, int site) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, bars, st, site));
}

// A rendezvous of several warps on an mbarrier (one arrival per warp), bounded
// like every other wait so that a warp that gave up cannot strand the others.
__device__ __forceinline__ bool warps_sync(uint64_t* bar, uint32_t parity, Bars* bars,
                                           DeviceStatus* st) {
  __syncwarp();
  if (threadIdx.x % 32 == 0) mbar_arrive(bar);
  return warp_wait(bar, parity, bars, st, kSiteFull);
}

// 16-byte chunk cc of row `row` in a tile of 128-byte swizzled regions of `reg` bytes.
__device__ __forceinline__ int swz(int row, int cc, int reg) {
  return (cc / 8) * reg + row * 128 + (((cc % 8) ^ (row % 8)) * 16);
}

template <typename T>
__device__ __forceinline__ uint4 pack8(const uint32_t* r, float mul) {
  uint4 o;
  o.x = tc::pack2<T>(__uint_as_float(r[0]) * mul, __uint_as_float(r[1]) * mul);
  o.y = tc::pack2<T>(__uint_as_float(r[2]) * mul, __uint_as_float(r[3]) * mul);
  o.z = tc::pack2<T>(__uint_as_float(r[4]) * mul, __uint_as_float(r[5]) * mul);
  o.w = tc::pack2<T>(__uint_as_float(r[6]) * mul, __uint_as_float(r[7]) * mul);
  return o;
}

// pack8 with the multiply two lanes per instruction (the same products)
template <typename T>
__device__ __forceinline__ uint4 pack8_x2(const uint32_t* r, float mul) {
  const unsigned long long m2 = tc::f2_pack(mul, mul);
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo, hi;
    tc::f2_unpack(tc::f2_mul(tc::f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                             m2),
                  lo, hi);
    h[i] = tc::pack2<T>(lo, hi);
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}

// Cache element C: the activation type T, or 8-bit E4M3 (bf16 activations).
// E4M3 rows of the host cache land in a staging slot of the stationary tile
// (the part of row r that the converted row r overwrites last) and are
// converted in place: K to T for the Q.K^T MMA, V to fp16 for P.V.
template <typename C>
constexpr bool kE4M3 = sizeof(C) == 1;

// Byte offset, inside one K or V tile, of the E4M3 staging slot of row r: the
// last 128-byte region of the row for D = 128, the upper 64 bytes of its
// single region for D = 64.  Converting row r reads the whole slot before it
// writes row r, and no other row's output touches it.
template <int D>
__device__ __forceinline__ int e4m3_slot(int r) {
  return (D / 64 - 1) * kRegKV + r * 128 + (D == 64 ? 64 : 0);
}

// Eight E4M3 values (the low 8 bytes of `w`, lower address first) as T or fp16 bits.
template <typename T>
__device__ __forceinline__ uint4 e4m3x8_to(uint2 w) {
  const uint32_t in[2] = {w.x, w.y};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t two = (in[i / 2] >> (16 * (i % 2))) & 0xFFFFu;
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
    if constexpr (std::is_same<T, __half>::value) {
      o[i] = (uint32_t)h.x | ((uint32_t)h.y << 16);
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
      o[i] = tc::pack2<T>(f.x, f.y);   // exact: E4M3 values are bf16 values
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// CTA u's unit: (b, KV head, Q tile group, chunk), chunks fastest.  That is
// the order in which a Q-stationary kernel would stream them (the naive
// baseline), and the fused prefill's order unless new_first.
// Where the units holding new tokens fit in one wave (new_first), they run
// first.  They are the longest (their projection comes before their tiles),
// so they stay out of the last wave; they read no cached rows, so fewer CTAs
// of the first wave queue for the link; and their unequal lengths stagger the
// starts of the prefix units after them.  Within each part the units run
// (b, KV head)-major with the chunks ascending, so that the units resident at
// one time share a KV head's Q tiles in L2.  The last nsplit prefix units
// run as two CTAs each (half of the Q tiles each, the chunk fetched by both),
// so that the last wave ends in shorter pieces.  tpg: Q tiles per CTA.
__device__ __forceinline__ void unit_of(int u, const TcArgs& a, int& c, int& tg, int& bh,
                                        int& tpg) {
  tpg = a.tiles_per_group;
  if (a.tile_groups != 1 || !a.new_first) {
    c = u % a.nchunks;
    tg = (u / a.nchunks) % a.tile_groups;
    bh = u / (a.nchunks * a.tile_groups);
    return;
  }
  tg = 0;
  int n1 = 0, n2 = 0;  // units holding new tokens (chunk >= the one holding key len[b]), others
  for (int b = 0; b < a.B; ++b) {
    const int cn = min(a.len[b] / kC, a.nchunks);
    n1 += a.Hkv * (a.nchunks - cn);
    n2 += a.Hkv * cn;
  }
  const bool first = u < n1;
  int r = first ? u : u - n1;
  if (!first && r >= n2 - a.nsplit) {  // a split unit: two consecutive CTAs
    const int j = r - (n2 - a.nsplit);
    r = n2 - a.nsplit + j / 2;
    tg = j % 2;
    tpg = (a.tiles_per_group + 1) / 2;
  }
  for (int b = 0; b < a.B; ++b) {
    const int cn = min(a.len[b] / kC, a.nchunks);  // first chunk with a new key
    const int n = first ? a.nchunks - cn : cn;     // this part's chunks per KV head
    if (r < a.Hkv * n) {
      bh = b * a.Hkv + r / n;
      c = (first ? cn : 0) + r % n;
      return;
    }
    r -= a.Hkv * n;
  }
  bh = 0;
  c = a.nchunks;  // not reached for u < B * Hkv * nchunks; a chunk past every key exits
}

template <typename T, typename C, int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_x,
                      const __grid_constant__ CUtensorMap map_wk,
                      const __grid_constant__ CUtensorMap map_wv,
                      const __grid_constant__ CUtensorMap map_po, const TcArgs a) {
  using Cfg = TcCfg<D>;
  constexpr int DR = Cfg::DR;
  constexpr int TQ = kBQ / G;  // tokens per Q tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  {
    // the 128-byte swizzle needs 1024-byte aligned tiles; if the padding that
    // takes does not fit in what was launched, report it and touch nothing
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    const uint32_t pad = (uint32_t)(smem - smem_raw);
    if (pad + Cfg::kOffBar + sizeof(Bars) > dyn) {
      if (threadIdx.x == 0) record_timeout(a.status, kSiteGridBarrier);
      return;
    }
  }
  uint8_t* ks = smem + Cfg::kOffK;
  uint8_t* vs = smem + Cfg::kOffV;
  uint8_t* qs = smem + Cfg::kOffQ;
  uint8_t* os = smem + Cfg::kOffO;
  Bars* bars = reinterpret_cast<Bars*>(smem + Cfg::kOffBar);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int c, tg, bh, tpg;
  unit_of(blockIdx.x, a, c, tg, bh, tpg);
  const int kvh = bh % a.Hkv, b = bh / a.Hkv;
  const int P = a.len[b];
  const int S = P + a.T;
  const int k0 = c * kC;
  if (k0 >= S) return;  // uniform over the CTA, before any barrier
  const int nkeys = min(kC, S - k0);
  const int nhost = max(0, min(kC, P - k0));   // rows [0, nhost) come from the host cache
  const bool has_new = k0 + kC > P;            // rows [nhost, C) are projected here
  const int pass0 = nhost / 128;               // first 128-row projection pass with new rows
  const int npass = has_new ? 2 - pass0 : 0;
  const int t_vis = max(0, k0 - P);            // first token that sees this chunk
  const int tile0 = tg * tpg;                  // this CTA's first Q tile of the chunk
  if (tile0 * TQ >= a.T - t_vis) return;       // uniform, before any barrier
  const int t_lo = t_vis + tile0 * TQ;         // first token of this CTA's tiles
  const int ntiles = min((a.T - t_lo + TQ - 1) / TQ, tpg);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars->pr_full[i], 1);
      mbar_init(&bars->pr_empty[i], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&bars->s_full[g], 1);
      mbar_init(&bars->p_full[g], 4);
      mbar_init(&bars->o_full[g], 1);
      mbar_init(&bars->r_free[g], 4);
    }
    for (int q = 0; q < 4; ++q) mbar_init(&bars->st_free[q], 1);
    mbar_init(&bars->kv_host, 32);
    mbar_init(&bars->kv_ready, 8);
    for (int p = 0; p < 2; ++p) {
      mbar_init(&bars->pr_done[p], 1);
      mbar_init(&bars->ap_sync[0][p], 4);
      mbar_init(&bars->ap_sync[1][p], 4);
    }
    mbar_init(&bars->pr_all, 1);
    mbar_init(&bars->vsync, 4);
    mbar_init(&bars->mma_drain, 1);
    bars->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tc::tmem_alloc(&bars->tmem_base, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const int nk_proj = (a.H + 63) / 64;  // TMA zero-fills past H

  if (warp == 0) {
    // ================================================================ loader
    // (a) cached rows of the chunk: host -> shared, 16-byte cp.async, swizzled.
    {
      const C* kg = static_cast<const C*>(a.k_read);
      const C* vg = static_cast<const C*>(a.v_read);
      constexpr int EPC = 16 / sizeof(C);  // elements per 16-byte chunk
      constexpr int CPR = D / EPC;         // 16-byte chunks per row
      const int rows = has_new ? nhost : kC;  // zero-fill the tail when nothing is projected
      for (int i = lane; i < rows * CPR; i += 32) {
        const int r = i / CPR, cc = i % CPR;
        const int off = kE4M3<C> ? e4m3_slot<D>(r) + cc * 16 : swz(r, cc, kRegKV);
        const bool ok = r < nhost;
        const size_t src = ok ? a.lay.row(b, kvh, k0 + r, D) + cc * EPC : 0;
        cp_async16(ks + off, kg + src, ok ? 16 : 0);
        cp_async16(vs + off, vg + src, ok ? 16 : 0);
      }
      // (the test hook withholds this arrival: every role's bounded wait then
      // gives up, a timeout is recorded and the combine writes NaN)
      if (!a.debug_withhold) cp_async_arrive_noinc(&bars->kv_host);
    }
    if (lane == 0) {
      // last load issued into each projection stage / Q buffer (-1: none)
      int last_g[4] = {-1, -1, -1, -1}, last_q[2] = {-1, -1};
      tc::prefetch_tmap(&map_q);
      // (b) projection operands, one 128-row pass at a time: x rows, [Wk | Wv]
      if (has_new) {
        tc::prefetch_tmap(&map_x);
        tc::prefetch_tmap(&map_wk);
        tc::prefetch_tmap(&map_wv);
        for (int ps = 0; ps < npass; ++ps) {
          const int xrow = b * a.T + (k0 + (pass0 + ps) * 128 - P);  // may be negative: zeros
          for (int kb = 0; kb < nk_proj; ++kb) {
            const int g = ps * nk_proj + kb;
            const int s = g % Cfg::SP;
            if (!wait_or_abort(&bars->pr_empty[s], ((g / Cfg::SP) & 1) ^ 1, bars, a.status,
                               kSiteEmpty))
              break;
            uint8_t* pa = qs + s * Cfg::kProjStage;
            uint8_t* pb = pa + Cfg::kProjA;
            tc::mbar_expect_tx(&bars->pr_full[s], Cfg::kProjStage);
            last_g[s] = g;
            tc::tma_load_2d(pa, &map_x, kb * 64, xrow, &bars->pr_full[s]);
#pragma unroll
            for (int r = 0; r < DR; ++r) {
              tc::tma_load_2d(pb + r * 8192, &map_wk, kvh * D + r * 64, kb * 64,
                              &bars->pr_full[s]);
              tc::tma_load_2d(pb + (DR + r) * 8192, &map_wv, kvh * D + r * 64, kb * 64,
                              &bars->pr_full[s]);
            }
          }
        }
        // the Q buffers alias the projection staging: wait until every pass
        // has consumed it
        wait_or_abort(&bars->pr_all, 0, bars, a.status, kSiteFull);
      }
      // (c) Q tiles, double-buffered
      for (int i = 0; i < ntiles && !bars->abort; ++i) {
        const int s = i & 1;
        if (!wait_or_abort(&bars->q_empty[s], ((i >> 1) & 1) ^ 1, bars, a.status, kSiteEmpty))
          break;
        const int tok = b * a.T + t_lo + i * TQ;
        tc::mbar_expect_tx(&bars->q_full[s], Cfg::kQ);
        last_q[s] = i;
#pragma unroll
        for (int r = 0; r < DR; ++r)
          tc::tma_load_3d(qs + s * Cfg::kQ + r * kRegQ, &map_q, r * 64, kvh * G, tok,
                          &bars->q_full[s]);
      }
      if (bars->abort) {
        // after a give-up nobody consumes the loads still in flight: let the
        // last one into each buffer land before the CTA leaves (bounded)
        for (int s = 0; s < Cfg::SP; ++s)
          if (last_g[s] >= 0) mbar_wait_drain(&bars->pr_full[s], (last_g[s] / Cfg::SP) & 1);
        for (int s = 0; s < 2; ++s)
          if (last_q[s] >= 0) mbar_wait_drain(&bars->q_full[s], (last_q[s] >> 1) & 1);
      }
    }
    cp_async_wait_all();
  } else if (warp == 1) {
    // ================================================================= MMA
    if (lane == 0) {
      const bool bf = DT<T>::code == DKV_BF16;
      // projection passes: [128 x H] . [H x 2D] -> TMEM columns [2D p, 2D p + 2D)
      // for pass p (2 passes x 2D <= 512 columns), so pass 1 runs while the
      // epilogue warps read pass 0 out
      if (has_new) {
        const uint32_t idesc = tc::idesc_f16(bf, 128, 2 * D, false, true);
        for (int ps = 0; ps < npass && !bars->abort; ++ps) {
          const uint32_t acc = tmem + (uint32_t)(ps * 2 * D);
          for (int kb = 0; kb < nk_proj; ++kb) {
            const int g = ps * nk_proj + kb;
            const int s = g % Cfg::SP;
            if (!wait_or_abort(&bars->pr_full[s], (g / Cfg::SP) & 1, bars, a.status, kSiteFull))
              break;
            tc::fence_after_sync();
            const uint32_t pa = smem_u32(qs + s * Cfg::kProjStage);
            const uint32_t pb = pa + Cfg::kProjA;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_ss(acc, tc::sdesc_sw128(pa + kk * 32, 16, 1024),
                         tc::sdesc_sw128(pb + kk * 2048, 8192, 1024), idesc, (kb | kk) != 0);
            tc::mma_commit(&bars->pr_empty[s]);
          }
          tc::mma_commit(&bars->pr_done[ps]);
        }
        tc::mma_commit(&bars->pr_all);  // arrives once every MMA above has completed
      }
      // the stationary K/V tile is complete (host rows landed, new rows written)
      wait_or_abort(&bars->kv_ready, 0, bars, a.status, kSiteFull);
      tc::fence_after_sync();
      const uint32_t idesc_s = tc::idesc_f16(bf, 128, kC, false, false);  // Q.K^T, N = 256
      const uint32_t idesc_o = tc::idesc_f16(false, 128, D, false, true); // P.V in fp16
      const uint32_t ka = smem_u32(ks), va = smem_u32(vs);
      // S of tile i into region i & 1 (its Q tile has landed; the region's
      // previous tile has had its O read out)
      auto issue_s = [&](int i) {
        const uint32_t rg = tmem + (uint32_t)(i & 1) * kTmRegion;
        const uint32_t qa = smem_u32(qs + (i & 1) * Cfg::kQ);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss(rg, tc::sdesc_sw128(qa + (kk / 4) * kRegQ + (kk % 4) * 32, 16, 1024),
                     tc::sdesc_sw128(ka + (kk / 4) * kRegKV + (kk % 4) * 32, 16, 1024), idesc_s,
                     kk != 0);
        tc::mma_commit(&bars->s_full[i & 1]);
        tc::mma_commit(&bars->q_empty[i & 1]);
      };
      // O of tile i = P.V, P read from the region's TMEM (fp16), V from shared
      auto issue_pv = [&](int i) {
        const uint32_t rg = tmem + (uint32_t)(i & 1) * kTmRegion;
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          tc::mma_ts(rg + kTmO, rg + kTmP + kk * 8,
                     tc::sdesc_sw128(va + kk * 2048, kRegKV, 1024), idesc_o, kk != 0);
        tc::mma_commit(&bars->o_full[i & 1]);
      };
      // Issue whichever is ready: the next S (tiles in order, at most two in
      // flight) or the next P.V (in order, once its softmax wrote P).  The
      // tests never suspend, so a barrier that is not ready cannot hold up one
      // that is.  Each test is on the phase right after one this thread has
      // already seen complete, so a parity test cannot mistake an older phase
      // for it.
      int ns = 0, np = 0;
      uint64_t deadline = 0;
      bool idle = false;
      while (np < ntiles) {
        bool did = false;
        if (ns < ntiles && ns < np + 2 &&
            mbar_test_wait(&bars->q_full[ns & 1], (ns >> 1) & 1) &&
            (ns < 2 || mbar_test_wait(&bars->r_free[ns & 1], ((ns - 2) >> 1) & 1))) {
          tc::fence_after_sync();
          issue_s(ns++);
          did = true;
        }
        if (np < ns && mbar_test_wait(&bars->p_full[np & 1], (np >> 1) & 1)) {
          tc::fence_after_sync();
          issue_pv(np++);
          did = true;
        }
        if (did) {
          idle = false;
          continue;
        }
        if (bars->abort) break;
        const uint64_t now = global_timer_ns();
        if (!idle) {
          idle = true;
          deadline = now + kWaitBudgetNs;
        } else if (now > deadline) {
          record_timeout(a.status, kSiteFull);
          bars->abort = 1;
          break;
        }
      }
      if (bars->abort) {
        // after a give-up, the MMAs already issued finish before TMEM is freed
        tc::mma_commit(&bars->mma_drain);
        mbar_wait_drain(&bars->mma_drain, 0);
      }
    }
    __syncwarp();
  } else {
    // ============================================= softmax / epilogue warps
    const int hh = (warp - 2) / 4;            // group: K/V half of the projection, tile parity
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;      // tile row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;

    // (a) projection epilogue per pass: half 0 takes the K columns, half 1
    //     the V columns; round, write into the stationary tile, append.
    for (int ps = 0; ps < npass; ++ps) {
      const bool ok = warp_wait(&bars->pr_done[ps], 0, bars, a.status, kSiteFull);
      tc::fence_after_sync();
      if (!ok) break;
      const int r = (pass0 + ps) * 128 + row;  // key row within the chunk
      const int key = k0 + r;
      const bool mine = r >= nhost;            // this row is a new key projected here
      const bool append = mine && key < S && tg == 0;  // appended once per chunk
      uint8_t* tile = hh ? vs : ks;
      C* const host_kv = static_cast<C*>(hh ? a.v_host : a.k_host);
      // (the row is looked up only where it exists: key < S)
      C* host = (kE4M3<C> && append) ? host_kv + a.lay.row(b, kvh, key, D) : nullptr;
#pragma unroll 1
      for (int part = 0; part < D / 32; ++part) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + lane_off + (uint32_t)(ps * 2 * D + hh * D + part * 32), v);
        tc::tmem_wait_ld();
        if constexpr (kE4M3<C>) {
          // the fp32 sums rounded once to E4M3 (nearest, saturating) are the
          // appended row; the tile holds those values (K as T, V as fp16)
          uint32_t e[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(
                make_float2(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1])),
                __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(
                make_float2(__uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])),
                __NV_SATFINITE, __NV_E4M3);
            e[q] = lo | (hi << 16);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint2 w = make_uint2(e[2 * q], e[2 * q + 1]);
            const uint4 o = hh ? e4m3x8_to<__half>(w) : e4m3x8_to<T>(w);
            if (mine) *reinterpret_cast<uint4*>(tile + swz(r, part * 4 + q, kRegKV)) = o;
          }
          if (append) {  // the append: 32 bytes
            reinterpret_cast<uint4*>(host + part * 32)[0] = make_uint4(e[0], e[1], e[2], e[3]);
            reinterpret_cast<uint4*>(host + part * 32)[1] = make_uint4(e[4], e[5], e[6], e[7]);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 o = pack8<T>(v + q * 8, 1.f);
            if (mine) *reinterpret_cast<uint4*>(tile + swz(r, part * 4 + q, kRegKV)) = o;
          }
        }
      }
      if constexpr (!kE4M3<C>) {
        // the append, from the tile once the half's four warps have written
        // the pass: consecutive threads take consecutive 16-byte pieces of a
        // row, so each warp writes whole 128-byte lines of the host cache (a
        // thread per row would leave every line to eight partial writes)
        if (tg == 0) {
          if (!warps_sync(&bars->ap_sync[hh][ps], 0, bars, a.status)) break;
          constexpr int CPR = D / 8;  // 16-byte pieces per row
          const int lo = max(nhost, (pass0 + ps) * 128);
          const int hi = min((pass0 + ps + 1) * 128, nkeys);
          const int ht = ((warp - 2) % 4) * 32 + lane;  // thread of the half
          for (int i = ht; i < (hi - lo) * CPR; i += 128) {
            const int rr = lo + i / CPR, cc = i % CPR;
            *reinterpret_cast<uint4*>(host_kv + a.lay.row(b, kvh, k0 + rr, D) + cc * 8) =
                *reinterpret_cast<const uint4*>(tile + swz(rr, cc, kRegKV));
          }
        }
      }
    }
    // the host rows have landed (loader's cp.async tracked by kv_host)
    wait_or_abort(&bars->kv_host, 0, bars, a.status, kSiteFull);
    if constexpr (kE4M3<C>) {
      // E4M3 host rows [0, nhost): group 0 converts K to T, group 1 V to
      // fp16, one row per thread and pass, from the row's staging slot.  No
      // chunk scale: E4M3 magnitudes stay below 448.
      uint8_t* tile = hh ? vs : ks;
#pragma unroll 1
      for (int rr = 0; rr < 2; ++rr) {
        const int r = rr * 128 + row;
        if (r >= nhost) break;
        uint4 in[D / 16];
#pragma unroll
        for (int cc = 0; cc < D / 16; ++cc)
          in[cc] = *reinterpret_cast<const uint4*>(tile + e4m3_slot<D>(r) + cc * 16);
#pragma unroll
        for (int cc = 0; cc < D / 16; ++cc) {
          const uint2 w0 = make_uint2(in[cc].x, in[cc].y), w1 = make_uint2(in[cc].z, in[cc].w);
          *reinterpret_cast<uint4*>(tile + swz(r, 2 * cc, kRegKV)) =
              hh ? e4m3x8_to<__half>(w0) : e4m3x8_to<T>(w0);
          *reinterpret_cast<uint4*>(tile + swz(r, 2 * cc + 1, kRegKV)) =
              hh ? e4m3x8_to<__half>(w1) : e4m3x8_to<T>(w1);
        }
      }
      if (hh == 1 && warp == 6 && lane == 0 && tg == 0)
        a.part_k[(size_t)c * a.B * a.Hkv + bh] = 0;
    } else if (hh == 1) {
      // P.V runs in fp16 (P keeps 11 significant bits).  For bf16 inputs the
      // stationary V chunk is converted to fp16 in place, times 2^-k with k the
      // smallest power making max|V| < 2^15 (k = 0 unless V is huge); the
      // chunk's partials carry that factor and the combine undoes it exactly.
      int k = 0;
      if constexpr (DT<T>::code == DKV_BF16) {
        float vmax = 0.f;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
          for (int cc = 0; cc < D / 8; ++cc) {
            const uint4 u = *reinterpret_cast<const uint4*>(vs + swz(rr * 128 + row, cc, kRegKV));
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = DT<T>::to_f2(w4[e]);
              vmax = fmaxf(vmax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
        }
        for (int off = 16; off > 0; off >>= 1)
          vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
        if (lane == 0) bars->vmax[quarter] = vmax;
        warps_sync(&bars->vsync, 0, bars, a.status);
        vmax = fmaxf(fmaxf(bars->vmax[0], bars->vmax[1]), fmaxf(bars->vmax[2], bars->vmax[3]));
        int e2 = 0;
        (void)frexpf(vmax, &e2);  // vmax < 2^e2
        k = (vmax == vmax && e2 > 15) ? e2 - 15 : 0;
        const float sc = exp2f((float)-k);
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
          for (int cc = 0; cc < D / 8; ++cc) {
            uint4* p16 = reinterpret_cast<uint4*>(vs + swz(rr * 128 + row, cc, kRegKV));
            const uint4 u = *p16;
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
            uint32_t h4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = DT<T>::to_f2(w4[e]);
              h4[e] = tc::pack2<__half>(f.x * sc, f.y * sc);
            }
            *p16 = make_uint4(h4[0], h4[1], h4[2], h4[3]);
          }
        }
      }
      if (warp == 6 && lane == 0 && tg == 0) a.part_k[(size_t)c * a.B * a.Hkv + bh] = k;
    }
    tc::fence_proxy_async_smem();  // generic/cp.async smem writes -> tensor core reads
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->kv_ready);

    // (b) the Q tiles.  Group hh takes tiles hh, hh + 2, ... in TMEM region
    //     hh; each thread owns one row (its TMEM lane) and all 256 scores of
    //     it, so a group needs no exchange beyond its four-warp arrivals.
    const float scale = a.scale_log2;
    const size_t TG = (size_t)a.T * G;
    const size_t blk = ((size_t)c * a.B + b) * a.Hkv + kvh;
    const uint32_t rg = tmem + lane_off + (uint32_t)hh * kTmRegion;
    // the storer hands its staging rows to the other group once its TMA store
    // has read them; it checks that while waiting for its next S, where the
    // warp would wait anyway
    bool pend = false;
    for (int j = hh, n = 0; j < ntiles; j += 2, ++n) {
      const uint32_t ph = n & 1;
      if (!warp_wait(&bars->s_full[hh], ph, bars, a.status, kSiteFull)) break;
      if (pend) {
        tc::bulk_wait_read_all();
        mbar_arrive(&bars->st_free[quarter]);
        pend = false;
      }
      tc::fence_after_sync();
      const int t_first = t_lo + j * TQ;
      // every key of the chunk is visible to every row of this tile
      const bool full = nkeys == kC && P + t_first >= k0 + kC - 1;
      const int t = t_first + row / G;
      const int nvis = min(nkeys, P + t - k0 + 1);  // keys [0, nvis) are visible to this row
      // P = 2^(s*scale - m) in fp16, 64 keys at a time, written over scores
      // this thread has already read (keys 2c, 2c+1 in column c).  m is the
      // max of the first 64 visible scores.  A later piece whose weights sum
      // to at most 2^14 has none above 2^14, which fp16 P and the fp32 sums
      // hold; one that sums to more (a score more than 8 above m, or an
      // overflow) takes its own max as m and rescales the weights already
      // written.  So m never exceeds the row max (the largest weight is >= 1)
      // and no weight ends up less precise than with the exact max.  l sums
      // the weights before the rounding: the normalisation then differs from
      // the rounded weights' sum by at most 2^-12 relative.
      constexpr float kSumBound = 16384.f;
      float mx = -INFINITY;
      float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int pc = 0; pc < kC / 64; ++pc) {
        uint32_t r[64];
        tc::tmem_ld32(rg + pc * 64, *reinterpret_cast<uint32_t(*)[32]>(r));
        tc::tmem_ld32(rg + pc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tc::tmem_wait_ld();
        // max of the piece's visible scores (scaled): the reference m for the
        // first piece, and in the rare rescale below
        auto piece_max = [&]() {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          if (full) {
#pragma unroll
            for (int k2 = 0; k2 < 64; ++k2)
              m4[k2 % 4] = fmaxf(m4[k2 % 4], __uint_as_float(r[k2]));
          } else {
#pragma unroll
            for (int k2 = 0; k2 < 64; ++k2)
              if (pc * 64 + k2 < nvis) m4[k2 % 4] = fmaxf(m4[k2 % 4], __uint_as_float(r[k2]));
          }
          return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * scale;
        };
        if (pc == 0) mx = piece_max();
        uint32_t w[32];
        float ls8[8];
        // (two keys per instruction: s*scale - m and the sums as fp32 pairs;
        // the sums ls8[2q], ls8[2q + 1] are pair q of the accumulators)
        auto weights = [&]() {
          const unsigned long long sc2 = tc::f2_pack(scale, scale), nm2 = tc::f2_pack(-mx, -mx);
          unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};  // +0.0f pairs
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k2 = pc * 64 + 2 * e;
            float p0, p1;
            tc::f2_unpack(tc::f2_fma(tc::f2_pack(__uint_as_float(r[2 * e]),
                                                 __uint_as_float(r[2 * e + 1])),
                                     sc2, nm2),
                          p0, p1);
            p0 = tc::ex2_approx(p0);
            p1 = tc::ex2_approx(p1);
            if (!full) {
              p0 = k2 < nvis ? p0 : 0.f;
              p1 = k2 + 1 < nvis ? p1 : 0.f;
            }
            w[e] = tc::pack2<__half>(p0, p1);
            acc[e % 4] = tc::f2_add(acc[e % 4], tc::f2_pack(p0, p1));
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) tc::f2_unpack(acc[q], ls8[2 * q], ls8[2 * q + 1]);
        };
        weights();
        if (pc > 0) {
          const float ls = ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
          const bool need = !(ls <= kSumBound);  // also an inf or NaN sum
          if (__any_sync(0xffffffffu, need)) {  // rare; TMEM access is warp-wide
            const float pm = need ? piece_max() : mx;
            const float f = need ? tc::ex2_approx(mx - pm) : 1.f;
            tc::tmem_wait_st();
            for (int q = 0; q < pc; ++q) {
              uint32_t v2[32];
              tc::tmem_ld32(rg + kTmP + q * 32, v2);
              tc::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&v2[e]));
                v2[e] = tc::pack2<__half>(v.x * f, v.y * f);
              }
              tc::tmem_st32(rg + kTmP + q * 32, v2);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) l8[q] *= f;
            mx = pm;
            weights();  // this piece again, against the new m
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) l8[q] += ls8[q];
        tc::tmem_st32(rg + kTmP + pc * 32, w);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[hh]);  // P is ready for the P.V MMA
      const float l = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));

      // epilogue: O / l in fp16 staged in shared memory and written with TMA
      // stores, the base-2 lse with plain stores; both land tile-contiguous:
      // block (c, b, kvh), rows (t, g)
      if (!warp_wait(&bars->o_full[hh], ph, bars, a.status, kSiteFull)) break;
      tc::fence_after_sync();
      uint32_t o[D];
#pragma unroll
      for (int part = 0; part < D / 32; ++part)
        tc::tmem_ld32(rg + kTmO + part * 32, *reinterpret_cast<uint32_t(*)[32]>(o + part * 32));
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->r_free[hh]);  // the region may take tile j + 2
      const float inv = 1.f / l;
      // the staging rows of this quarter have been read by tile j - 1's store
      if (j > 0 && !warp_wait(&bars->st_free[quarter], (j - 1) & 1, bars, a.status, kSiteEmpty))
        break;
#pragma unroll
      for (int q = 0; q < D / 8; ++q)
        *reinterpret_cast<uint4*>(os + swz(row, q, kRegQ)) = pack8_x2<__half>(o + q * 8, inv);
      if (t < a.T) a.part_lse[blk * TG + (size_t)t * G + row % G] = mx + log2f(l);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int row0 = t_first * G + quarter * 32;  // rows past T*G are clipped by the store
        if (row0 < (int)TG) {
#pragma unroll
          for (int rr = 0; rr < DR; ++rr)
            tc::tma_store_3d(&map_po, rr * 64, row0, (int)blk, os + rr * kRegQ + quarter * 32 * 128);
          tc::bulk_commit();
        }
      }
      pend = lane == 0;
    }
    if (pend) {
      tc::bulk_wait_read_all();
      mbar_arrive(&bars->st_free[quarter]);
    }
    if (lane == 0) tc::bulk_wait_all();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// out[b,t,h,:] = sum_c w_c 2^k_c o'_c / sum_c w_c, w_c = 2^(lse_c - max lse),
// over the chunks c = 0 .. (len+t)/C that row sees, in one pass with a running
// max (what is accumulated is rescaled when a chunk's lse exceeds it).  D/16
// threads per row, each owning 16 consecutive outputs: two 16-byte loads of
// the fp16 partials per chunk (32 contiguous bytes per thread).  If a wait of
// the fused kernel gave up (the status word holds an error), the outputs are
// NaN rather than a merge of partials that were never written.
template <typename T, int D>
__global__ void __launch_bounds__(128) prefill_combine_tc_kernel(
    const __half* __restrict__ part_o, const float* __restrict__ part_lse,
    const int* __restrict__ part_k, T* __restrict__ out, LenArray len, int B, int T_, int Hq,
    int Hkv, const DeviceStatus* status) {
  constexpr int TPR = D / 16;           // threads per row
  constexpr int RPB = 128 / TPR;        // rows per block
  const size_t R = (size_t)B * T_ * Hq;
  const int sub = threadIdx.x % TPR;
  size_t row = (size_t)blockIdx.x * RPB + threadIdx.x / TPR;
  const bool active = row < R;
  if (!active) row = R - 1;
  const int h = row % Hq;
  const int bt = row / Hq;
  const int t = bt % T_, b = bt / T_;
  const int G = Hq / Hkv;
  const int kh = b * Hkv + h / G;
  // partial row of (b, t, h) inside each chunk's R rows: block (b, kvh), row (t, g)
  const size_t pr = (size_t)kh * T_ * G + (size_t)t * G + h % G;
  const int last = (len.v[b] + t) / kC;
  if (*(const volatile int*)&status->code != 0) {
    if (active) {
      uint32_t nan[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) nan[e] = __float_as_uint(NAN);
      uint4* dst = reinterpret_cast<uint4*>(out + row * D) + 2 * sub;
      dst[0] = pack8<T>(nan, 1.f);
      dst[1] = pack8<T>(nan + 8, 1.f);
    }
    return;
  }
  float M = -INFINITY;
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  float den = 0.f;
#pragma unroll 2
  for (int c = 0; c <= last; ++c) {
    const float lc = __ldg(part_lse + c * R + pr);
    if (lc > M) {  // new running max: rescale what is accumulated (0 at the start)
      const float sc = exp2f(M - lc);
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] *= sc;
      den *= sc;
      M = lc;
    }
    const float w = exp2f(lc - M);
    const float wk = ldexpf(w, __ldg(part_k + (size_t)c * B * Hkv + kh));
    const uint4* src = reinterpret_cast<const uint4*>(part_o + (c * R + pr) * D) + 2 * sub;
    const uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
    const uint32_t w8[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w8[e]));
      acc[2 * e] = fmaf(wk, f.x, acc[2 * e]);
      acc[2 * e + 1] = fmaf(wk, f.y, acc[2 * e + 1]);
    }
    den += w;
  }
  if (active) {
    const float inv = 1.f / den;
    uint32_t r[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(acc[e]);
    uint4* dst = reinterpret_cast<uint4*>(out + row * D) + 2 * sub;
    dst[0] = pack8<T>(r, inv);
    dst[1] = pack8<T>(r + 8, inv);
  }
}

template <typename T, typename C, int D, int G>
cudaError_t launch_t(const TcArgs& args, const CUtensorMap& mq, const CUtensorMap& mx,
                     const CUtensorMap& mk, const CUtensorMap& mv, void* out, cudaStream_t s,
                     const KernelTimer& timer) {
  auto k = prefill_tc_kernel<T, C, D, G>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_request<D>());
  if (e != cudaSuccess) return e;
  CUtensorMap mpo;
  if (!make_tmap_partial(&mpo, args.part_o, D, (uint64_t)args.T * G,
                         (uint64_t)args.nchunks * args.B * args.Hkv))
    return cudaErrorInvalidValue;
  const int units = args.B * args.Hkv * args.nchunks * args.tile_groups + args.nsplit;
  timer.before(s);
  k<<<units, kThreads, smem_request<D>(), s>>>(mq, mx, mk, mv, mpo, args);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  timer.after(s);
  LenArray len;
  for (int i = 0; i < kMaxBatch; ++i) len.v[i] = args.len[i];
  const size_t R = (size_t)args.B * args.T * args.Hq;
  constexpr int RPB = 128 / (D / 16);
  prefill_combine_tc_kernel<T, D><<<(unsigned)((R + RPB - 1) / RPB), 128, 0, s>>>(
      static_cast<const __half*>(args.part_o), args.part_lse, args.part_k, static_cast<T*>(out),
      len, args.B, args.T, args.Hq, args.Hkv, args.status);
  return cudaGetLastError();
}

}  // namespace

int prefill_tc_chunk_keys() { return kC; }

bool prefill_supported(int dtype, int D, int G) {
  return (dtype == DKV_BF16 || dtype == DKV_FP16) && (D == 64 || D == 128) &&
         (G == 1 || G == 2 || G == 4 || G == 8);
}

cudaError_t launch_prefill_tc(const PrefillParams& p, int dtype, const void* wq, cudaStream_t s,
                              int* launches, const KernelTimer& timer) {
  const int G = p.Hq / p.Hkv;
  const int D = p.D;
  if (p.H % 8 != 0 || !prefill_supported(dtype, D, G)) return cudaErrorInvalidValue;
  // 1. Q projection (HBM-resident Q) on the tensor cores
  cudaError_t e = launch_gemm_tc(p.x, wq, const_cast<void*>(p.q), p.B * p.T, p.Hq * D, p.H,
                                 dtype, p.status, s);
  if (e != cudaSuccess) return e;
  // 2. fused KV projection + append + KV-stationary attention, 3. combine
  CUtensorMap mq, mx, mk, mv;
  if (!make_tmap_q(&mq, p.q, dtype, D, p.Hq, (uint64_t)p.B * p.T, G, kBQ / G) ||
      !make_tmap_2d(&mx, p.x, dtype, (uint64_t)p.B * p.T, p.H, 64, kBQ) ||
      !make_tmap_2d(&mk, p.wk, dtype, p.H, (uint64_t)p.Hkv * D, 64, 64) ||
      !make_tmap_2d(&mv, p.wv, dtype, p.H, (uint64_t)p.Hkv * D, 64, 64))
    return cudaErrorInvalidValue;
  TcArgs a;
  a.k_read = p.k_read; a.v_read = p.v_read; a.k_host = p.k_host; a.v_host = p.v_host;
  a.part_o = p.part_o; a.part_lse = p.part_lse; a.part_k = p.part_k; a.status = p.status;
  a.B = p.B; a.T = p.T; a.H = p.H; a.Hq = p.Hq; a.Hkv = p.Hkv; a.lay = p.lay;
  a.nchunks = p.nchunks; a.scale_log2 = p.scale_log2;
  const int tiles = (p.T + kBQ / G - 1) / (kBQ / G);  // Q tiles of the longest chunk
  a.tiles_per_group = p.naive ? 1 : tiles;
  a.debug_withhold = p.debug_withhold;
  a.tile_groups = p.naive ? tiles : 1;
  // New-token units first where they fit in one wave of CTAs (one per SM).
  // Otherwise (many new chunks against the prefix: the fp16 MHA prefill has
  // a quarter of its units new) the link would idle while wave after wave
  // only projects, and the plain order, which mixes the two kinds, is faster.
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  long long nnew = 0;
  for (int b = 0; b < p.B; ++b)
    nnew += (long long)p.Hkv * (p.nchunks - std::min(p.len[b] / kC, p.nchunks));
  a.new_first = !p.naive && nnew <= sms;
  // and, where a prefix unit is long (64 Q tiles or more), the last wave's
  // worth of prefix units split in two.  Each split unit fetches its chunk
  // twice (at most one more chunk per SM over the link) and waits for the
  // cached rows twice, which a unit of a few dozen tiles does not repay.
  const long long nprefix = (long long)p.B * p.Hkv * p.nchunks - nnew;
  a.nsplit = a.new_first && tiles >= 64 ? (int)std::min<long long>(sms, nprefix) : 0;
  for (int i = 0; i < kMaxBatch; ++i) a.len[i] = p.len[i];
#define DKV_TC(TT, DD, GG) \
  if (D == DD && G == GG) e = launch_t<TT, TT, DD, GG>(a, mq, mx, mk, mv, p.out, s, timer); else
#define DKV_TC8(DD, GG) \
  if (D == DD && G == GG) \
    e = launch_t<__nv_bfloat16, __nv_fp8_e4m3, DD, GG>(a, mq, mx, mk, mv, p.out, s, timer); else
  if (p.kv_fp8) {
    if (dtype != DKV_BF16) return cudaErrorInvalidValue;
    DKV_TC8(64, 1) DKV_TC8(64, 2) DKV_TC8(64, 4) DKV_TC8(64, 8)
    DKV_TC8(128, 1) DKV_TC8(128, 2) DKV_TC8(128, 4) DKV_TC8(128, 8) e = cudaErrorInvalidValue;
  } else if (dtype == DKV_BF16) {
    DKV_TC(__nv_bfloat16, 64, 1) DKV_TC(__nv_bfloat16, 64, 2) DKV_TC(__nv_bfloat16, 64, 4)
    DKV_TC(__nv_bfloat16, 64, 8) DKV_TC(__nv_bfloat16, 128, 1) DKV_TC(__nv_bfloat16, 128, 2)
    DKV_TC(__nv_bfloat16, 128, 4) DKV_TC(__nv_bfloat16, 128, 8) e = cudaErrorInvalidValue;
  } else {
    DKV_TC(__half, 64, 1) DKV_TC(__half, 64, 2) DKV_TC(__half, 64, 4) DKV_TC(__half, 64, 8)
    DKV_TC(__half, 128, 1) DKV_TC(__half, 128, 2) DKV_TC(__half, 128, 4) DKV_TC(__half, 128, 8)
    e = cudaErrorInvalidValue;
  }
#undef DKV_TC
#undef DKV_TC8
  if (e == cudaSuccess && launches) *launches += 3;
  return e;
}

}  // namespace dkv
