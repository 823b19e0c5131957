// Fused KV-stationary prefill on the 5th-generation tensor cores.
//
// DirectKV's prefill holds each (K, V) tile fetched from host memory
// stationary and iterates over the HBM-resident Q ("Paper Notes: DirectKV",
// System Architecture, Attention Fusion Engine; Key Ideas (1)); the K/V
// projection of new tokens is fused so the fresh K/V are produced on chip and
// consumed there (Key Ideas (2)); warps specialise into loading, computing and
// storing roles (Key Ideas (3)).
//
// One CTA = one unit (sequence b, KV head, chunk of C = 128 keys).
//   1. The chunk's K and V land in shared memory (128-byte swizzled rows):
//      cached rows with 16-byte cp.async from the mapped host cache (each host
//      byte crosses the link once), new rows from a tcgen05 GEMM
//      [x rows] . [Wk | Wv] (TMA-fed, accumulator in TMEM) whose epilogue
//      rounds them, writes them into the stationary tile and appends them to
//      the host cache.
//   2. Every Q tile of the KV group that can see the chunk (128 rows = 128/G
//      tokens x G heads, TMA from HBM) runs S = Q.K^T (tcgen05, TMEM), a
//      complete softmax over the chunk (it is stationary, so there is no
//      running rescale), O = P.V (tcgen05, TMEM, fp16 operands), and its
//      normalised O and base-2 log-sum-exp are written as the chunk's
//      partial.  Two softmax warpgroups take alternate Q tiles, each with its
//      own S and O in TMEM and its own P tile in shared memory, so the tensor
//      cores run one group's MMAs while the other group does its softmax.
// A combine kernel merges the chunks' partials per query row.
//
// Warp roles (320 threads): warp 0 loads (TMA / cp.async), warp 1 allocates
// TMEM and issues every MMA from one thread, warps 2-5 and 6-9 are the two
// softmax / epilogue groups (one TMEM lane = one row per thread).  Every wait
// is bounded.
#include "tc_common.cuh"

namespace dkv {

bool make_tmap_2d(CUtensorMap* map, const void* base, int dtype, uint64_t rows, uint64_t cols,
                  uint32_t box_cols, uint32_t box_rows);
bool make_tmap_q(CUtensorMap* map, const void* q, int dtype, int D, int Hq, uint64_t tokens,
                 int G, int TQ);
bool make_tmap_partial(CUtensorMap* map, void* base, int D, uint64_t rows, uint64_t blocks);

namespace {

constexpr int kC = 128;        // keys per stationary chunk
constexpr int kBQ = 128;       // rows per Q tile
constexpr int kThreads = 320;  // 10 warps
constexpr int kRegion = 128 * 128;  // one 128-row x 128-byte swizzled region

template <int D>
struct TcCfg {
  static constexpr int DR = D / 64;                    // 128-byte regions per row
  static constexpr int kKV = kC * D * 2;               // one of K or V
  static constexpr int kQ = kBQ * D * 2;               // one Q tile
  static constexpr int kP = kBQ * kC * 2;              // one P tile
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKV;
  static constexpr int kOffQ = kOffV + kKV;            // two Q buffers
  static constexpr int kOffP = kOffQ + 2 * kQ;         // two P buffers
  static constexpr int kOffBar = kOffP + 2 * kP;
  // projection staging (aliases the Q and P buffers): x block [128 x 64] and
  // W block [64 x 2D], two stages
  static constexpr int kProjA = kBQ * 64 * 2;          // 16 KB
  static constexpr int kProjB = 64 * 2 * D * 2;        // 16 / 32 KB
  static constexpr int kProjStage = kProjA + kProjB;
  static_assert(2 * kProjStage <= 2 * kQ + 2 * kP, "projection staging must fit");
  static constexpr int kSmem = 1024 + kOffBar + 256;
};

struct Bars {
  uint64_t q_full[2], q_empty[2], s_full[2], s_empty[2], p_full[2], p_empty[2], o_full[2],
      o_empty[2], kv_host, kv_ready, pr_full[2], pr_empty[2], pr_done;
  uint32_t tmem_base;
  volatile int abort;
  float vmax[4];
};

struct TcArgs {
  const void* k_read;
  const void* v_read;
  void* k_host;
  void* v_host;
  void* part_o;     // [nchunks, B*T*Hq, D] fp16, normalised, times 2^-k of the chunk
  float* part_lse;  // [nchunks, B*T*Hq]
  int* part_k;      // [nchunks, B*Hkv]
  DeviceStatus* status;
  int B, T, H, Hq, Hkv, S_max, nchunks;
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

// Warp-uniform bounded wait (tcgen05.ld after it needs the whole warp).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, Bars* bars,
                                          DeviceStatus* st, int site) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, bars, st, site));
}

__device__ __forceinline__ int swz_off(int row, int cc) {  // 16-byte chunk cc of a row
  return (cc / 8) * kRegion + row * 128 + (((cc % 8) ^ (row % 8)) * 16);
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

template <typename T, int D, int G>
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
  uint8_t* ks = smem + Cfg::kOffK;
  uint8_t* vs = smem + Cfg::kOffV;
  uint8_t* qs = smem + Cfg::kOffQ;
  uint8_t* ps = smem + Cfg::kOffP;
  Bars* bars = reinterpret_cast<Bars*>(smem + Cfg::kOffBar);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = blockIdx.x % a.nchunks;
  const int bh = blockIdx.x / a.nchunks;
  const int kvh = bh % a.Hkv, b = bh / a.Hkv;
  const int P = a.len[b];
  const int S = P + a.T;
  const int k0 = c * kC;
  if (k0 >= S) return;  // uniform over the CTA, before any barrier
  const int nkeys = min(kC, S - k0);
  const int nhost = max(0, min(kC, P - k0));   // rows [0, nhost) come from the host cache
  const bool has_new = k0 + kC > P;            // rows [P - k0, C) are projected here
  const int t_lo = max(0, k0 - P);             // first token that sees this chunk
  const int ntiles = (a.T - t_lo + TQ - 1) / TQ;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_empty[i], 4);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->p_empty[i], 1);
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->o_empty[i], 4);
      mbar_init(&bars->pr_full[i], 1);
      mbar_init(&bars->pr_empty[i], 1);
    }
    mbar_init(&bars->kv_host, 32);
    mbar_init(&bars->kv_ready, 8);
    mbar_init(&bars->pr_done, 1);
    bars->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tc::tmem_alloc(&bars->tmem_base, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  // TMEM columns: S[0] 0..127, S[1] 128..255, O[0] 256.., O[1] 384..; the
  // projection accumulator (2D columns) reuses 0..2D-1 before the Q loop.
  const int nk_proj = (a.H + 63) / 64;  // TMA zero-fills past H
  const size_t head_off = ((size_t)b * a.Hkv + kvh) * a.S_max * D;

  if (warp == 0) {
    // ================================================================ loader
    // (a) cached rows of the chunk: host -> shared, 16-byte cp.async, swizzled.
    {
      const T* kg = static_cast<const T*>(a.k_read) + head_off + (size_t)k0 * D;
      const T* vg = static_cast<const T*>(a.v_read) + head_off + (size_t)k0 * D;
      constexpr int CPR = D / 8;  // 16-byte chunks per row
      const int rows = has_new ? nhost : kC;  // zero-fill the tail when nothing is projected
      for (int i = lane; i < rows * CPR; i += 32) {
        const int r = i / CPR, cc = i % CPR;
        const int off = swz_off(r, cc);
        const bool ok = r < nhost;
        const size_t src = ok ? (size_t)r * D + cc * 8 : 0;
        cp_async16(ks + off, kg + src, ok ? 16 : 0);
        cp_async16(vs + off, vg + src, ok ? 16 : 0);
      }
      cp_async_arrive_noinc(&bars->kv_host);
    }
    if (lane == 0) {
      tc::prefetch_tmap(&map_q);
      // (b) projection operands for the new rows: x rows and [Wk | Wv] columns
      if (has_new) {
        tc::prefetch_tmap(&map_x);
        tc::prefetch_tmap(&map_wk);
        tc::prefetch_tmap(&map_wv);
        const int xrow = b * a.T + (k0 - P);  // may be negative: TMA fills zeros
        for (int kb = 0; kb < nk_proj; ++kb) {
          const int s = kb & 1;
          if (!wait_or_abort(&bars->pr_empty[s], ((kb >> 1) & 1) ^ 1, bars, a.status, kSiteEmpty))
            break;
          uint8_t* pa = qs + s * Cfg::kProjStage;
          uint8_t* pb = pa + Cfg::kProjA;
          tc::mbar_expect_tx(&bars->pr_full[s], Cfg::kProjStage);
          tc::tma_load_2d(pa, &map_x, kb * 64, xrow, &bars->pr_full[s]);
#pragma unroll
          for (int r = 0; r < DR; ++r) {
            tc::tma_load_2d(pb + r * 8192, &map_wk, kvh * D + r * 64, kb * 64, &bars->pr_full[s]);
            tc::tma_load_2d(pb + (DR + r) * 8192, &map_wv, kvh * D + r * 64, kb * 64,
                            &bars->pr_full[s]);
          }
        }
        // the Q buffers alias the projection staging: wait until it is consumed
        wait_or_abort(&bars->pr_done, 0, bars, a.status, kSiteFull);
      }
      // (c) Q tiles
      for (int i = 0; i < ntiles && !bars->abort; ++i) {
        const int s = i & 1;
        if (!wait_or_abort(&bars->q_empty[s], ((i >> 1) & 1) ^ 1, bars, a.status, kSiteEmpty))
          break;
        const int tok = b * a.T + t_lo + i * TQ;
        tc::mbar_expect_tx(&bars->q_full[s], Cfg::kQ);
#pragma unroll
        for (int r = 0; r < DR; ++r)
          tc::tma_load_3d(qs + s * Cfg::kQ + r * kRegion, &map_q, r * 64, kvh * G, tok,
                          &bars->q_full[s]);
      }
    }
    cp_async_wait_all();
  } else if (warp == 1) {
    // ================================================================= MMA
    if (lane == 0) {
      const bool bf = DT<T>::code == DKV_BF16;
      // projection: [128 x H] . [H x 2D] -> TMEM columns 0..2D-1
      if (has_new) {
        const uint32_t idesc = tc::idesc_f16(bf, 128, 2 * D, false, true);
        for (int kb = 0; kb < nk_proj; ++kb) {
          const int s = kb & 1;
          if (!wait_or_abort(&bars->pr_full[s], (kb >> 1) & 1, bars, a.status, kSiteFull)) break;
          tc::fence_after_sync();
          const uint32_t pa = smem_u32(qs + s * Cfg::kProjStage);
          const uint32_t pb = pa + Cfg::kProjA;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_ss(tmem, tc::sdesc_sw128(pa + kk * 32, 16, 1024),
                       tc::sdesc_sw128(pb + kk * 2048, 8192, 1024), idesc, (kb | kk) != 0);
          tc::mma_commit(&bars->pr_empty[s]);
        }
        tc::mma_commit(&bars->pr_done);
      }
      // the stationary K/V tile is complete (host rows landed, new rows written)
      wait_or_abort(&bars->kv_ready, 0, bars, a.status, kSiteFull);
      tc::fence_after_sync();
      const uint32_t idesc_s = tc::idesc_f16(bf, 128, kC, false, false);  // Q.K^T
      const uint32_t idesc_o = tc::idesc_f16(false, 128, D, false, true); // P.V in fp16
      const uint32_t ka = smem_u32(ks), va = smem_u32(vs);
      auto issue_pv = [&](int j) {
        const int s = j & 1;
        if (!wait_or_abort(&bars->p_full[s], (j >> 1) & 1, bars, a.status, kSiteFull)) return;
        if (!wait_or_abort(&bars->o_empty[s], ((j >> 1) & 1) ^ 1, bars, a.status, kSiteEmpty))
          return;
        tc::fence_after_sync();
        const uint32_t pa = smem_u32(ps + s * Cfg::kP);
        const uint32_t o_tm = tmem + 256 + s * 128;
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          tc::mma_ss(o_tm, tc::sdesc_sw128(pa + (kk / 4) * kRegion + (kk % 4) * 32, 16, 1024),
                     tc::sdesc_sw128(va + kk * 2048, kRegion, 1024), idesc_o, kk != 0);
        tc::mma_commit(&bars->o_full[s]);
        tc::mma_commit(&bars->p_empty[s]);
      };
      for (int i = 0; i < ntiles && !bars->abort; ++i) {
        const int s = i & 1;
        if (!wait_or_abort(&bars->q_full[s], (i >> 1) & 1, bars, a.status, kSiteFull)) break;
        if (!wait_or_abort(&bars->s_empty[s], ((i >> 1) & 1) ^ 1, bars, a.status, kSiteEmpty))
          break;
        tc::fence_after_sync();
        const uint32_t qa = smem_u32(qs + s * Cfg::kQ);
        const uint32_t s_tm = tmem + s * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss(s_tm, tc::sdesc_sw128(qa + (kk / 4) * kRegion + (kk % 4) * 32, 16, 1024),
                     tc::sdesc_sw128(ka + (kk / 4) * kRegion + (kk % 4) * 32, 16, 1024), idesc_s,
                     kk != 0);
        tc::mma_commit(&bars->s_full[s]);
        tc::mma_commit(&bars->q_empty[s]);
        if (i > 0) issue_pv(i - 1);
      }
      if (ntiles > 0 && !bars->abort) issue_pv(ntiles - 1);
    }
    __syncwarp();
  } else {
    // ============================================ two softmax / epilogue groups
    const int grp = (warp - 2) / 4;           // group g takes tiles i with i % 2 == g
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;      // tile row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;

    // (a) projection epilogue: group 0 takes the K columns, group 1 the V
    //     columns; round, write into the stationary tile, append to the host.
    if (has_new) {
      const bool ok = warp_wait(&bars->pr_done, 0, bars, a.status, kSiteFull);
      tc::fence_after_sync();
      if (ok) {
        const int key = k0 + row;
        const bool mine = row >= P - k0;      // this row is a new key projected here
        const bool append = mine && key < S;
        uint8_t* tile = grp ? vs : ks;
        T* host = static_cast<T*>(grp ? a.v_host : a.k_host) + head_off + (size_t)key * D;
#pragma unroll 1
        for (int part = 0; part < D / 32; ++part) {
          uint32_t r[32];
          tc::tmem_ld32(tmem + lane_off + grp * D + part * 32, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 o = pack8<T>(r + v * 8, 1.f);
            if (mine) *reinterpret_cast<uint4*>(tile + swz_off(row, part * 4 + v)) = o;
            if (append) *reinterpret_cast<uint4*>(host + part * 32 + v * 8) = o;  // the append
          }
        }
      }
    }
    // the host rows have landed (loader's cp.async tracked by kv_host)
    wait_or_abort(&bars->kv_host, 0, bars, a.status, kSiteFull);
    if (grp == 1) {
      // P.V runs in fp16 (P keeps 11 significant bits).  For bf16 inputs the
      // stationary V chunk is converted to fp16 in place, times 2^-k with k the
      // smallest power making max|V| < 2^15 (k = 0 unless V is huge); the
      // chunk's partials carry that factor and the combine undoes it exactly.
      int k = 0;
      if constexpr (DT<T>::code == DKV_BF16) {
        float vmax = 0.f;
#pragma unroll
        for (int cc = 0; cc < D / 8; ++cc) {
          const uint4 u = *reinterpret_cast<const uint4*>(vs + swz_off(row, cc));
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = DT<T>::to_f2(w4[e]);
            vmax = fmaxf(vmax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
        for (int off = 16; off > 0; off >>= 1)
          vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
        if (lane == 0) bars->vmax[quarter] = vmax;
        named_bar_sync(2, 128);
        vmax = fmaxf(fmaxf(bars->vmax[0], bars->vmax[1]), fmaxf(bars->vmax[2], bars->vmax[3]));
        int e2 = 0;
        (void)frexpf(vmax, &e2);  // vmax < 2^e2
        k = (vmax == vmax && e2 > 15) ? e2 - 15 : 0;
        const float sc = exp2f((float)-k);
#pragma unroll
        for (int cc = 0; cc < D / 8; ++cc) {
          uint4* p16 = reinterpret_cast<uint4*>(vs + swz_off(row, cc));
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
      if (warp == 6 && lane == 0) a.part_k[(size_t)c * a.B * a.Hkv + bh] = k;
    }
    tc::fence_proxy_async_smem();  // generic/cp.async smem writes -> tensor core reads
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->kv_ready);

    // (b) this group's Q tiles: softmax, then the output epilogue
    const float scale = a.scale_log2;
    const int s = grp;
    const uint32_t s_tm = tmem + s * 128 + lane_off;
    const uint32_t o_tm = tmem + 256 + s * 128 + lane_off;
    uint8_t* prow = ps + s * Cfg::kP;
    const bool leader = warp == 2 + 4 * grp && lane == 0;  // issues this group's TMA stores
    // partials of this unit: block (c, b, kvh) of T*G rows ordered (token, head)
    const size_t TG = (size_t)a.T * G;
    const size_t blk = ((size_t)c * a.B + b) * a.Hkv + kvh;
    for (int i = grp; i < ntiles; i += 2) {
      const uint32_t ph = (i >> 1) & 1;
      if (!warp_wait(&bars->s_full[s], ph, bars, a.status, kSiteFull)) break;
      tc::fence_after_sync();
      const int t_first = t_lo + i * TQ;
      // every key of the chunk is visible to every row of this tile
      const bool full = nkeys == kC && P + t_first >= k0 + kC - 1;
      const int t = t_first + row / G;
      const int nvis = min(nkeys, P + t - k0 + 1);
      // the whole S row in registers: four TMEM loads in flight, one wait
      uint32_t r[kC];
#pragma unroll
      for (int part = 0; part < kC / 32; ++part)
        tc::tmem_ld32(s_tm + part * 32, *reinterpret_cast<uint32_t(*)[32]>(r + part * 32));
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_empty[s]);  // S may be overwritten by tile i + 2
      // row max of the visible raw scores (eight independent chains)
      float m8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) m8[q] = -INFINITY;
      if (full) {
#pragma unroll
        for (int j = 0; j < kC; ++j) m8[j % 8] = fmaxf(m8[j % 8], __uint_as_float(r[j]));
      } else {
#pragma unroll
        for (int j = 0; j < kC; ++j)
          if (j < nvis) m8[j % 8] = fmaxf(m8[j % 8], __uint_as_float(r[j]));
      }
      const float mraw = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const float mx = mraw * scale;
      // P = 2^(s*scale - m) in fp16; l sums the rounded weights so the P.V
      // product is normalised by exactly the weights it used.
      if (!warp_wait(&bars->p_empty[s], ph ^ 1, bars, a.status, kSiteEmpty)) break;
      // the P buffer also staged the previous tile's output: its TMA store
      // must have finished reading it
      if (i >= 2) {
        if (leader) tc::bulk_wait_read_all();
        named_bar_sync(3 + grp, 128);
      }
      float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int cc = 0; cc < kC / 8; ++cc) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = cc * 8 + 2 * e;
          float p0 = tc::ex2_approx(fmaf(__uint_as_float(r[j]), scale, -mx));
          float p1 = tc::ex2_approx(fmaf(__uint_as_float(r[j + 1]), scale, -mx));
          if (!full) {
            p0 = j < nvis ? p0 : 0.f;
            p1 = j + 1 < nvis ? p1 : 0.f;
          }
          w[e] = tc::pack2<__half>(p0, p1);
          const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          l8[2 * e] += back.x;
          l8[2 * e + 1] += back.y;
        }
        *reinterpret_cast<uint4*>(prow + swz_off(row, cc)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      const float l = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[s]);  // P is ready for the P.V MMA
      // epilogue of this tile: O / l in fp16 staged in the (consumed) P buffer
      // and written with TMA stores; the base-2 lse with plain stores.  Both
      // land tile-contiguous: block (c, b, kvh), rows (t, g).
      if (!warp_wait(&bars->o_full[s], ph, bars, a.status, kSiteFull)) break;
      tc::fence_after_sync();
      const float inv = 1.f / l;
#pragma unroll
      for (int part = 0; part < D / 32; ++part)
        tc::tmem_ld32(o_tm + part * 32, *reinterpret_cast<uint32_t(*)[32]>(r + part * 32));
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty[s]);  // O may be overwritten by tile i + 2
#pragma unroll
      for (int v = 0; v < D / 8; ++v)
        *reinterpret_cast<uint4*>(prow + swz_off(row, v)) = pack8<__half>(r + v * 8, inv);
      if (t < a.T) a.part_lse[blk * TG + (size_t)t * G + row % G] = mx + log2f(l);
      tc::fence_proxy_async_smem();
      named_bar_sync(3 + grp, 128);
      if (leader) {
#pragma unroll
        for (int rg = 0; rg < DR; ++rg)
          tc::tma_store_3d(&map_po, rg * 64, t_first * G, (int)blk, prow + rg * kRegion);
        tc::bulk_commit();
      }
    }
    if (leader) tc::bulk_wait_all();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// out[b,t,h,:] = sum_c w_c 2^k_c o'_c / sum_c w_c, w_c = 2^(lse_c - max lse),
// over the chunks c = 0 .. (len+t)/C that row sees.  D/8 threads per row, each
// owning 8 consecutive outputs (16-byte loads of the fp16 partials).
template <typename T, int D>
__global__ void __launch_bounds__(128) prefill_combine_tc_kernel(
    const __half* __restrict__ part_o, const float* __restrict__ part_lse,
    const int* __restrict__ part_k, T* __restrict__ out, LenArray len, int B, int T_, int Hq,
    int Hkv) {
  constexpr int TPR = D / 8;            // threads per row
  constexpr int RPB = 128 / TPR;        // rows per block
  const size_t R = (size_t)B * T_ * Hq;
  const int sub = threadIdx.x % TPR;
  size_t row = (size_t)blockIdx.x * RPB + threadIdx.x / TPR;
  const bool active = row < R;
  if (!active) row = R - 1;             // keep every lane in the shuffles
  const int h = row % Hq;
  const int bt = row / Hq;
  const int t = bt % T_, b = bt / T_;
  const int G = Hq / Hkv;
  const int kh = b * Hkv + h / G;
  // partial row of (b, t, h) inside each chunk's R rows: block (b, kvh), row (t, g)
  const size_t pr = (size_t)kh * T_ * G + (size_t)t * G + h % G;
  const int last = (len.v[b] + t) / kC;
  float M = -INFINITY;
  for (int c = sub; c <= last; c += TPR) M = fmaxf(M, __ldg(part_lse + c * R + pr));
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float den = 0.f;
#pragma unroll 4
  for (int c = 0; c <= last; ++c) {
    const float w = exp2f(__ldg(part_lse + c * R + pr) - M);
    const float wk = ldexpf(w, __ldg(part_k + (size_t)c * B * Hkv + kh));
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(part_o + (c * R + pr) * D) + sub);
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
      acc[2 * e] = fmaf(wk, f.x, acc[2 * e]);
      acc[2 * e + 1] = fmaf(wk, f.y, acc[2 * e + 1]);
    }
    den += w;
  }
  if (active) {
    const float inv = 1.f / den;
    uint32_t r[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(acc[e]);
    reinterpret_cast<uint4*>(out + row * D)[sub] = pack8<T>(r, inv);
  }
}

template <typename T, int D, int G>
cudaError_t launch_t(const TcArgs& args, const CUtensorMap& mq, const CUtensorMap& mx,
                     const CUtensorMap& mk, const CUtensorMap& mv, void* out, cudaStream_t s,
                     const KernelTimer& timer) {
  auto k = prefill_tc_kernel<T, D, G>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  CUtensorMap mpo;
  if (!make_tmap_partial(&mpo, args.part_o, D, (uint64_t)args.T * G,
                         (uint64_t)args.nchunks * args.B * args.Hkv))
    return cudaErrorInvalidValue;
  const int units = args.B * args.Hkv * args.nchunks;
  timer.before(s);
  k<<<units, kThreads, TcCfg<D>::kSmem, s>>>(mq, mx, mk, mv, mpo, args);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  timer.after(s);
  LenArray len;
  for (int i = 0; i < kMaxBatch; ++i) len.v[i] = args.len[i];
  const size_t R = (size_t)args.B * args.T * args.Hq;
  constexpr int RPB = 128 / (D / 8);
  prefill_combine_tc_kernel<T, D><<<(unsigned)((R + RPB - 1) / RPB), 128, 0, s>>>(
      static_cast<const __half*>(args.part_o), args.part_lse, args.part_k, static_cast<T*>(out),
      len, args.B, args.T, args.Hq, args.Hkv);
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
  a.B = p.B; a.T = p.T; a.H = p.H; a.Hq = p.Hq; a.Hkv = p.Hkv; a.S_max = p.S_max;
  a.nchunks = p.nchunks; a.scale_log2 = p.scale_log2;
  for (int i = 0; i < kMaxBatch; ++i) a.len[i] = p.len[i];
#define DKV_TC(TT, DD, GG) \
  if (D == DD && G == GG) e = launch_t<TT, DD, GG>(a, mq, mx, mk, mv, p.out, s, timer); else
  if (dtype == DKV_BF16) {
    DKV_TC(__nv_bfloat16, 64, 1) DKV_TC(__nv_bfloat16, 64, 2) DKV_TC(__nv_bfloat16, 64, 4)
    DKV_TC(__nv_bfloat16, 64, 8) DKV_TC(__nv_bfloat16, 128, 1) DKV_TC(__nv_bfloat16, 128, 2)
    DKV_TC(__nv_bfloat16, 128, 4) DKV_TC(__nv_bfloat16, 128, 8) e = cudaErrorInvalidValue;
  } else {
    DKV_TC(__half, 64, 1) DKV_TC(__half, 64, 2) DKV_TC(__half, 64, 4) DKV_TC(__half, 64, 8)
    DKV_TC(__half, 128, 1) DKV_TC(__half, 128, 2) DKV_TC(__half, 128, 4) DKV_TC(__half, 128, 8)
    e = cudaErrorInvalidValue;
  }
#undef DKV_TC
  if (e == cudaSuccess && launches) *launches += 3;
  return e;
}

}  // namespace dkv
