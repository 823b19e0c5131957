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
//      running rescale), O = P.V (tcgen05, TMEM), and its normalised O and
//      base-2 log-sum-exp are written as the chunk's partial.  S, O, P and the
//      Q tile are double-buffered so the tensor cores work on tile i+1 while
//      the softmax warps finish tile i.
// A combine kernel merges the chunks' partials per query row.
//
// Warp roles (192 threads): warp 0 loads (TMA / cp.async), warp 1 allocates
// TMEM and issues every MMA from one thread, warps 2-5 run the projection
// epilogue, the softmax and the output epilogue (one TMEM lane = one row per
// thread).  Every wait is bounded.
#include <mutex>

#include "tc_common.cuh"

namespace dkv {

bool make_tmap_2d(CUtensorMap* map, const void* base, int dtype, uint64_t rows, uint64_t cols,
                  uint32_t box_cols, uint32_t box_rows);
bool make_tmap_q(CUtensorMap* map, const void* q, int dtype, int D, int Hq, uint64_t tokens,
                 int G, int TQ);

namespace {

constexpr int kC = 128;        // keys per stationary chunk
constexpr int kBQ = 128;       // rows per Q tile
constexpr int kThreads = 192;  // 6 warps
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

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_x,
                      const __grid_constant__ CUtensorMap map_wk,
                      const __grid_constant__ CUtensorMap map_wv, const TcArgs a) {
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
    mbar_init(&bars->kv_ready, 4);
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
  const uint32_t tm_s[2] = {tmem, tmem + 128};
  const uint32_t tm_o[2] = {tmem + 256, tmem + 384};
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
        const int off = (cc / 8) * kRegion + r * 128 + (((cc % 8) ^ (r % 8)) * 16);
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
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          tc::mma_ss(tm_o[s], tc::sdesc_sw128(pa + (kk / 4) * kRegion + (kk % 4) * 32, 16, 1024),
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
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss(tm_s[s], tc::sdesc_sw128(qa + (kk / 4) * kRegion + (kk % 4) * 32, 16, 1024),
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
    // ==================================================== softmax / epilogue
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;      // tile row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // (a) projection epilogue: round, write into the stationary tile, append
    if (has_new) {
      const bool ok = __all_sync(0xffffffffu,
                                 wait_or_abort(&bars->pr_done, 0, bars, a.status, kSiteFull));
      tc::fence_after_sync();
      const int key = k0 + row;
      if (ok) {  // warp-uniform: every lane runs the TMEM loads
        const bool mine = row >= P - k0;  // this row is a new key projected here
        T* kh = static_cast<T*>(a.k_host) + head_off + (size_t)key * D;
        T* vh = static_cast<T*>(a.v_host) + head_off + (size_t)key * D;
        const bool append = mine && key < S;
#pragma unroll 1
        for (int part = 0; part < 2 * D / 32; ++part) {  // K columns, then V columns
          uint32_t r[32];
          tc::tmem_ld32(tmem + lane_off + part * 32, r);
          tc::tmem_wait_ld();
          const bool isv = part >= D / 32;
          const int d0 = (part % (D / 32)) * 32;
          uint8_t* tile = isv ? vs : ks;
          T* host = isv ? vh : kh;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 o;
            o.x = tc::pack2<T>(__uint_as_float(r[v * 8 + 0]), __uint_as_float(r[v * 8 + 1]));
            o.y = tc::pack2<T>(__uint_as_float(r[v * 8 + 2]), __uint_as_float(r[v * 8 + 3]));
            o.z = tc::pack2<T>(__uint_as_float(r[v * 8 + 4]), __uint_as_float(r[v * 8 + 5]));
            o.w = tc::pack2<T>(__uint_as_float(r[v * 8 + 6]), __uint_as_float(r[v * 8 + 7]));
            const int cc = (d0 + v * 8) / 8;  // 16-byte chunk index in the row
            if (mine)
              *reinterpret_cast<uint4*>(tile + (cc / 8) * kRegion + row * 128 +
                                        (((cc % 8) ^ (row % 8)) * 16)) = o;
            if (append) *reinterpret_cast<uint4*>(host + d0 + v * 8) = o;  // the append
          }
        }
      }
    }
    // the host rows have landed (loader's cp.async tracked by kv_host)
    wait_or_abort(&bars->kv_host, 0, bars, a.status, kSiteFull);
    // P.V runs in fp16 (P keeps 11 significant bits).  For bf16 inputs the
    // stationary V chunk is converted to fp16 in place, times 2^-k with k the
    // smallest power making max|V| < 2^15 (k = 0 unless V is huge); the
    // chunk's partials carry that factor and the combine undoes it exactly.
    {
      int k = 0;
      if constexpr (DT<T>::code == DKV_BF16) {
        uint8_t* vrow = vs;  // this thread's row: key `row`
        float vmax = 0.f;
#pragma unroll
        for (int cc = 0; cc < D / 8; ++cc) {
          const uint4 u = *reinterpret_cast<const uint4*>(
              vrow + (cc / 8) * kRegion + row * 128 + (((cc % 8) ^ (row % 8)) * 16));
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
        named_bar_sync(1, 128);
        vmax = fmaxf(fmaxf(bars->vmax[0], bars->vmax[1]), fmaxf(bars->vmax[2], bars->vmax[3]));
        int e2 = 0;
        (void)frexpf(vmax, &e2);  // vmax < 2^e2
        k = (vmax == vmax && e2 > 15) ? e2 - 15 : 0;
        const float sc = exp2f((float)-k);
#pragma unroll
        for (int cc = 0; cc < D / 8; ++cc) {
          uint4* p16 = reinterpret_cast<uint4*>(vrow + (cc / 8) * kRegion + row * 128 +
                                                 (((cc % 8) ^ (row % 8)) * 16));
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
      if (threadIdx.x == 64) a.part_k[(size_t)c * a.B * a.Hkv + bh] = k;
    }
    tc::fence_proxy_async_smem();  // generic/cp.async smem writes -> tensor core reads
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->kv_ready);

    // (b) Q tiles: softmax of tile i, then the output epilogue of tile i-1
    float m_prev = 0.f, l_prev = 1.f;
    int t_prev = 0;
    const float scale = a.scale_log2;
    auto epilogue = [&](int j, float m, float l, bool live) {
      const int s = j & 1;
      const bool ok = __all_sync(0xffffffffu, wait_or_abort(&bars->o_full[s], (j >> 1) & 1, bars,
                                                            a.status, kSiteFull));
      tc::fence_after_sync();
      if (!ok) return;
      const int t = t_lo + j * TQ + row / G;
      const int h = kvh * G + row % G;
      const size_t grow = ((size_t)b * a.T + t) * a.Hq + h;
      const size_t slot = (size_t)c * ((size_t)a.B * a.T * a.Hq) + grow;
      const float inv = 1.f / l;
      __half* po = static_cast<__half*>(a.part_o) + slot * D;
#pragma unroll 1
      for (int part = 0; part < D / 32; ++part) {
        uint32_t r[32];
        tc::tmem_ld32(tm_o[s] + lane_off + part * 32, r);
        tc::tmem_wait_ld();
        if (live && t < a.T) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 o;
            o.x = tc::pack2<__half>(__uint_as_float(r[v * 8 + 0]) * inv, __uint_as_float(r[v * 8 + 1]) * inv);
            o.y = tc::pack2<__half>(__uint_as_float(r[v * 8 + 2]) * inv, __uint_as_float(r[v * 8 + 3]) * inv);
            o.z = tc::pack2<__half>(__uint_as_float(r[v * 8 + 4]) * inv, __uint_as_float(r[v * 8 + 5]) * inv);
            o.w = tc::pack2<__half>(__uint_as_float(r[v * 8 + 6]) * inv, __uint_as_float(r[v * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(po + part * 32 + v * 8) = o;
          }
        }
      }
      if (live && t < a.T) a.part_lse[slot] = m + log2f(l);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty[s]);
    };

    for (int i = 0; i < ntiles; ++i) {
      const int s = i & 1;
      const bool ok = __all_sync(0xffffffffu, wait_or_abort(&bars->s_full[s], (i >> 1) & 1, bars,
                                                            a.status, kSiteFull));
      tc::fence_after_sync();
      if (!ok) break;
      const int t = t_lo + i * TQ + row / G;
      const int qpos = P + t;
      const int nvis = min(nkeys, qpos - k0 + 1);  // keys 0..nvis-1 visible to this row
      float sv[kC];
#pragma unroll
      for (int part = 0; part < kC / 32; ++part) {
        uint32_t r[32];
        tc::tmem_ld32(tm_s[s] + lane_off + part * 32, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[part * 32 + j] = __uint_as_float(r[j]);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_empty[s]);  // S buffer may be overwritten
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kC; ++j) {
        sv[j] = j < nvis ? sv[j] * scale : -INFINITY;
        mx = fmaxf(mx, sv[j]);
      }
      // P = 2^(s - m) rounded to the dtype; l sums the rounded values so the
      // P.V product is normalised by exactly the weights it used.
      if (!__all_sync(0xffffffffu, wait_or_abort(&bars->p_empty[s], ((i >> 1) & 1) ^ 1, bars,
                                                 a.status, kSiteEmpty)))
        break;
      uint8_t* prow = ps + s * Cfg::kP;
      float l = 0.f;
#pragma unroll
      for (int cc = 0; cc < kC / 8; ++cc) {  // 16-byte chunks of the P row
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = exp2f(sv[cc * 8 + 2 * e] - mx);
          const float p1 = exp2f(sv[cc * 8 + 2 * e + 1] - mx);
          w[e] = tc::pack2<__half>(p0, p1);
          const float2 back = DT<__half>::to_f2(w[e]);
          l += back.x + back.y;
        }
        *reinterpret_cast<uint4*>(prow + (cc / 8) * kRegion + row * 128 +
                                  (((cc % 8) ^ (row % 8)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[s]);
      if (i > 0) epilogue(i - 1, m_prev, l_prev, true);
      m_prev = mx;
      l_prev = l;
      t_prev = t;
    }
    (void)t_prev;
    if (ntiles > 0 && !bars->abort) epilogue(ntiles - 1, m_prev, l_prev, true);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// out[b,t,h,:] = sum_c w_c 2^k_c o'_c / sum_c w_c, w_c = 2^(lse_c - max lse),
// over the chunks c = 0 .. (len+t)/C that row sees.
template <typename T>
__global__ void prefill_combine_tc_kernel(const __half* __restrict__ part_o,
                                          const float* __restrict__ part_lse,
                                          const int* __restrict__ part_k, T* __restrict__ out,
                                          LenArray len, int B, int T_, int Hq, int Hkv, int D,
                                          int C) {
  const size_t row = blockIdx.x;  // (b*T + t)*Hq + h
  const int h = row % Hq;
  const int bt = row / Hq;
  const int t = bt % T_, b = bt / T_;
  const int kh = b * Hkv + h / (Hq / Hkv);
  const int last = (len.v[b] + t) / C;
  const size_t R = (size_t)B * T_ * Hq;
  float M = -INFINITY;
  for (int c = 0; c <= last; ++c) M = fmaxf(M, part_lse[c * R + row]);
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float num = 0.f, den = 0.f;
    for (int c = 0; c <= last; ++c) {
      const float w = exp2f(part_lse[c * R + row] - M);
      const float o = __half2float(part_o[(c * R + row) * D + d]);
      num = fmaf(w * exp2f((float)part_k[(size_t)c * B * Hkv + kh]), o, num);
      den += w;
    }
    out[row * D + d] = DT<T>::from_f(num / den);
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
  const int units = args.B * args.Hkv * args.nchunks;
  timer.before(s);
  k<<<units, kThreads, TcCfg<D>::kSmem, s>>>(mq, mx, mk, mv, args);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  timer.after(s);
  LenArray len;
  for (int i = 0; i < kMaxBatch; ++i) len.v[i] = args.len[i];
  prefill_combine_tc_kernel<T><<<args.B * args.T * args.Hq, D, 0, s>>>(
      static_cast<const __half*>(args.part_o), args.part_lse, args.part_k, static_cast<T*>(out),
      len, args.B, args.T, args.Hq, args.Hkv, D, kC);
  return cudaGetLastError();
}

}  // namespace

int prefill_tc_chunk_keys() { return kC; }

// Q viewed as [tokens][Hq][D]: box (64 of D) x (G heads) x (128/G tokens).
bool make_tmap_q(CUtensorMap* map, const void* q, int dtype, int D, int Hq, uint64_t tokens,
                 int G, int TQ);

cudaError_t launch_prefill_tc(const PrefillParams& p, int dtype, const void* wq, cudaStream_t s,
                              int* launches, const KernelTimer& timer) {
  const int G = p.Hq / p.Hkv;
  const int D = p.D;
  if (p.H % 8 != 0 || (D != 64 && D != 128) || (G != 1 && G != 2 && G != 4 && G != 8))
    return cudaErrorInvalidValue;
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
