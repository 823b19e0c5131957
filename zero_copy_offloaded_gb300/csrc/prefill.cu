// Prefill (chunked prefill): Q projection to HBM, then the fused KV-stationary
// kernel, then the per-chunk combine.
//
// DirectKV's prefill strategy iterates over HBM-resident Q for each (K, V)
// tile fetched from host memory, treating the host tile as stationary and
// pushing the reload cost onto HBM ("Paper Notes: DirectKV", System
// Architecture, Attention Fusion Engine; Key Ideas (1)).  The K/V projection
// of the new tokens is fused so the fresh K/V stay in shared memory and are
// consumed there (Key Ideas (2)); the new rows are written to the host cache
// once (KV Cache Manager).
//
// Unit of work: (sequence b, KV head, chunk of C keys).  The chunk's K and V
// sit in shared memory for the whole unit: rows below the cached length are
// copied from the host cache with 16-byte cp.async (read across the link
// exactly once), rows in the new region are projected in place from x and
// appended to the host cache.  Every query row (token t, head g of the group)
// that can see the chunk (causal: position len+t >= chunk start) is then
// attended against it; a row's result over one chunk is complete, so it is
// written as a normalised partial (o, lse) and the combine merges chunks.
#include "dkv_internal.cuh"

namespace dkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kKC = 16;  // reduction rows per GEMM staging step

// ---------------------------------------------------------------------------
// Sequential-order SIMT GEMM tile: rows [r0, r0+ROWS) x columns of a
// [H, ldb] matrix block given by `col_ptr(c)` (c in [0, COLS)), reduced over
// j = 0..H-1 in order with one fp32 FMA chain per output.  Each thread owns an
// 8 x 8 micro-tile.  The epilogue gets (row, col, acc).
template <typename T, int COLS>
struct SeqGemm {
  static constexpr int kColGroups = COLS / 8;              // threads across columns
  static constexpr int kRowGroups = kThreads / kColGroups; // threads across rows
  static constexpr int kRows = kRowGroups * 8;
  static constexpr int kSmemBytes = 2 * (kRows * kKC + kKC * COLS) * 2;

  // A: rows of x ([*, H], row stride H); nrows valid rows starting at a_row0.
  // Bsrc(j, c) -> pointer to 8 contiguous T of the B block at row j, cols c..c+7.
  template <typename BPtr, typename Epi>
  __device__ static void run(const T* A, int H, int nrows, BPtr bptr, uint8_t* smem, Epi epi,
                             int ncols = COLS) {
    T* as = reinterpret_cast<T*>(smem);                 // [2][kRows][kKC]
    T* bs = as + 2 * kRows * kKC;                       // [2][kKC][COLS]
    const int tid = threadIdx.x;
    const int tr = tid / kColGroups, tc = tid % kColGroups;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    const int nsteps = H / kKC;
    auto issue = [&](int step, int buf) {
      const int j0 = step * kKC;
      // A tile: kRows x kKC (kKC = 16 -> two 16-byte pieces per row)
      for (int i = tid; i < kRows * 2; i += kThreads) {
        const int r = i / 2, pc = i % 2;
        const bool ok = r < nrows;
        cp_async16(as + (buf * kRows + r) * kKC + pc * 8,
                   A + (size_t)(ok ? r : 0) * H + j0 + pc * 8, ok ? 16 : 0);
      }
      for (int i = tid; i < kKC * kColGroups; i += kThreads) {
        const int j = i / kColGroups, cg = i % kColGroups;
        const bool ok = cg * 8 < ncols;  // ncols is a multiple of 8
        cp_async16(bs + (buf * kKC + j) * COLS + cg * 8, bptr(j0 + j, ok ? cg * 8 : 0), ok ? 16 : 0);
      }
      cp_async_commit();
    };
    issue(0, 0);
    for (int s = 0; s < nsteps; ++s) {
      if (s + 1 < nsteps) {
        issue(s + 1, (s + 1) & 1);
        cp_async_wait_group<1>();
      } else {
        cp_async_wait_group<0>();
      }
      __syncthreads();
      const T* a = as + (s & 1) * kRows * kKC;
      const T* b = bs + (s & 1) * kKC * COLS;
#pragma unroll 2
      for (int k = 0; k < kKC; ++k) {
        float av[8], bv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) av[i] = DT<T>::to_f(a[(tr * 8 + i) * kKC + k]);
        const uint4 bw = *reinterpret_cast<const uint4*>(b + k * COLS + tc * 8);
        float2 b0 = DT<T>::to_f2(bw.x), b1 = DT<T>::to_f2(bw.y);
        float2 b2 = DT<T>::to_f2(bw.z), b3 = DT<T>::to_f2(bw.w);
        bv[0] = b0.x; bv[1] = b0.y; bv[2] = b1.x; bv[3] = b1.y;
        bv[4] = b2.x; bv[5] = b2.y; bv[6] = b3.x; bv[7] = b3.y;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = tr * 8 + i;
      if (r < nrows && tc * 8 < ncols) {
#pragma unroll
        for (int j = 0; j < 8; ++j) epi(r, tc * 8 + j, acc[i][j]);
      }
    }
  }
};

// ---------------------------------------------------------------------------
template <int D>
struct PrefillCfg {
  static constexpr int kChunkBytes = 128 * 1024;          // K + V of one chunk
  static constexpr int C = kChunkBytes / (2 * D * 2);      // keys per chunk
  static constexpr int kRowBytes = D * 2;
  static constexpr int CPR = kRowBytes / 16;
  static constexpr int kProjCols = 2 * D;                  // K and V columns
  using Proj = SeqGemm<__nv_bfloat16, 2 * D>;              // sizes only (same for fp16)
  static constexpr int kQOff = kChunkBytes;                // per-warp q rows (fp32)
  static constexpr int kQBytes = kWarps * D * 4;
  static constexpr int kGemmOff = kQOff + kQBytes;
  static constexpr int kSmem = kGemmOff + Proj::kSmemBytes;
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads, 1) prefill_fused_kernel(const PrefillParams p) {
  using Cfg = PrefillCfg<D>;
  constexpr int C = Cfg::C;
  constexpr int CPR = Cfg::CPR;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ks = smem;                               // [C][D] swizzled
  uint8_t* vs = smem + C * D * 2;                   // [C][D] swizzled
  float* qw = reinterpret_cast<float*>(smem + Cfg::kQOff);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  const int u = blockIdx.x;
  const int c = u % p.nchunks;
  const int bh = u / p.nchunks;
  const int kvh = bh % p.Hkv, b = bh / p.Hkv;
  const int P = p.len[b];
  const int S = P + p.T;
  const int k0 = c * C;
  if (k0 >= S) return;
  const int k1 = min(k0 + C, S);
  const int nkeys = k1 - k0;

  // 1. stationary chunk, cached part: host rows [k0, min(k1, P)) read once
  const size_t head_off = ((size_t)b * p.Hkv + kvh) * p.S_max * D;
  {
    const T* kg = static_cast<const T*>(p.k_read) + head_off;
    const T* vg = static_cast<const T*>(p.v_read) + head_off;
    const int nhost = max(0, min(k1, P) - k0);
    for (int i = tid; i < nhost * CPR; i += kThreads) {
      const int row = i / CPR, cc = i % CPR;
      const int dst = row * (D * 2) + swz_chunk(row, cc) * 16;
      const size_t src = (size_t)(k0 + row) * D + cc * 8;
      cp_async16(ks + dst, kg + src, 16);
      cp_async16(vs + dst, vg + src, 16);
    }
    cp_async_commit();
  }
  // 2. stationary chunk, new part: project rows [max(k0, P), k1) in place and
  //    append them to the host cache.
  const int nfirst = max(k0, P);
  if (nfirst < k1) {
    using Proj = SeqGemm<T, 2 * D>;
    const T* wk = static_cast<const T*>(p.wk) + kvh * D;
    const T* wv = static_cast<const T*>(p.wv) + kvh * D;
    const int ldw = p.Hkv * D;
    T* kh = static_cast<T*>(p.k_host) + head_off;
    T* vh = static_cast<T*>(p.v_host) + head_off;
    auto bptr = [&](int j, int cc) {
      return cc < D ? wk + (size_t)j * ldw + cc : wv + (size_t)j * ldw + (cc - D);
    };
    for (int rb = nfirst; rb < k1; rb += Proj::kRows) {
      const int nr = min(Proj::kRows, k1 - rb);
      const T* xa = static_cast<const T*>(p.x) + ((size_t)b * p.T + (rb - P)) * p.H;
      auto epi = [&](int r, int cc, float v) {
        const T val = DT<T>::from_f(v);
        const int key = rb + r, row = key - k0;
        const int d = cc % D;
        uint8_t* tile = cc < D ? ks : vs;
        *reinterpret_cast<T*>(tile + row * (D * 2) + swz_chunk(row, d / 8) * 16 + (d % 8) * 2) = val;
        (cc < D ? kh : vh)[(size_t)key * D + d] = val;   // the append
      };
      Proj::run(xa, p.H, nr, bptr, smem + Cfg::kGemmOff, epi);
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // 3. every query row that sees this chunk: tokens t >= k0 - P, heads of the group
  const int t0 = max(0, k0 - P);
  const int nrows = (p.T - t0) * G;
  const T* qg = static_cast<const T*>(p.q);
  float* myq = qw + warp * D;
  constexpr int KPL = C / 32;          // keys per lane
  constexpr int DPL = D / 32;          // output dims per lane
  const size_t R_all = (size_t)p.B * p.T * p.Hq;
  for (int row = warp; row < nrows; row += kWarps) {
    const int t = t0 + row / G, g = row % G;
    const int h = kvh * G + g;
    const int qpos = P + t;
    const size_t qrow = ((size_t)b * p.T + t) * p.Hq + h;
    for (int d = lane; d < D; d += 32) myq[d] = DT<T>::to_f(qg[qrow * D + d]);
    __syncwarp();
    float s[KPL];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int n = lane + 32 * i;
      const int key = k0 + n;
      float dot = -INFINITY;
      if (n < nkeys && key <= qpos) {
        dot = 0.f;
        const uint8_t* kr = ks + n * (D * 2);
#pragma unroll 4
        for (int cc = 0; cc < CPR; ++cc) {
          const uint4 kv = *reinterpret_cast<const uint4*>(kr + swz_chunk(n, cc) * 16);
          const float* qq = myq + cc * 8;
          float2 a0 = DT<T>::to_f2(kv.x), a1 = DT<T>::to_f2(kv.y);
          float2 a2 = DT<T>::to_f2(kv.z), a3 = DT<T>::to_f2(kv.w);
          dot = fmaf(qq[0], a0.x, dot); dot = fmaf(qq[1], a0.y, dot);
          dot = fmaf(qq[2], a1.x, dot); dot = fmaf(qq[3], a1.y, dot);
          dot = fmaf(qq[4], a2.x, dot); dot = fmaf(qq[5], a2.y, dot);
          dot = fmaf(qq[6], a3.x, dot); dot = fmaf(qq[7], a3.y, dot);
        }
        dot *= p.scale_log2;
      }
      s[i] = dot;
      mx = fmaxf(mx, dot);
    }
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float l = 0.f;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      s[i] = exp2f(s[i] - mx);
      l += s[i];
    }
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    float o[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[j] = 0.f;
    const int nvis = min(nkeys, qpos - k0 + 1);
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int nbase = 32 * i;
      if (nbase >= nvis) break;
      const int lim = min(32, nvis - nbase);
      for (int src = 0; src < lim; ++src) {
        const float pw = __shfl_sync(0xffffffffu, s[i], src);
        const int n = nbase + src;
        const uint8_t* vr = vs + n * (D * 2);
#pragma unroll
        for (int j = 0; j < DPL; ++j) {
          const int d = lane + 32 * j;
          const T v = *reinterpret_cast<const T*>(vr + swz_chunk(n, d / 8) * 16 + (d % 8) * 2);
          o[j] = fmaf(pw, DT<T>::to_f(v), o[j]);
        }
      }
    }
    const size_t slot = (size_t)c * R_all + qrow;
    float* po = static_cast<float*>(p.part_o) + slot * D;
    const float inv = 1.f / l;
#pragma unroll
    for (int j = 0; j < DPL; ++j) po[lane + 32 * j] = o[j] * inv;
    if (lane == 0) p.part_lse[slot] = mx + log2f(l);
    __syncwarp();
  }
}

// out[b,t,h,:] = merge over chunks c = 0 .. (len+t)/C of the partials.
template <typename T>
__global__ void prefill_combine_kernel(const PrefillParams p, int C) {
  const size_t row = blockIdx.x;   // (b*T + t)*Hq + h
  const int h = row % p.Hq;
  const int bt = row / p.Hq;
  const int t = bt % p.T, b = bt / p.T;
  (void)h;
  const int last = (p.len[b] + t) / C;
  const size_t R_all = (size_t)p.B * p.T * p.Hq;
  float M = -INFINITY;
  for (int c = 0; c <= last; ++c) M = fmaxf(M, p.part_lse[c * R_all + row]);
  const float* po = static_cast<const float*>(p.part_o);
  for (int d = threadIdx.x; d < p.D; d += blockDim.x) {
    float num = 0.f, den = 0.f;
    for (int c = 0; c <= last; ++c) {
      const float w = exp2f(p.part_lse[c * R_all + row] - M);
      num = fmaf(w, po[(c * R_all + row) * p.D + d], num);
      den += w;
    }
    static_cast<T*>(p.out)[row * p.D + d] = DT<T>::from_f(num / den);
  }
}

template <typename T, int D, int G>
cudaError_t launch_prefill_t(const PrefillParams& p, cudaStream_t s, int* launches,
                             const void* wq, const KernelTimer& timer) {
  // 1. Q projection (HBM-resident Q) on the tensor cores
  {
    cudaError_t e = launch_gemm_tc(p.x, wq, const_cast<void*>(p.q), p.B * p.T, p.Hq * D, p.H,
                                   DT<T>::code, p.status, s);
    if (e != cudaSuccess) return e;
  }
  // 2. fused KV projection + append + KV-stationary attention
  {
    using Cfg = PrefillCfg<D>;
    auto kern = prefill_fused_kernel<T, D, G>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    const int units = p.B * p.Hkv * p.nchunks;
    timer.before(s);
    kern<<<units, kThreads, Cfg::kSmem, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    timer.after(s);
  }
  // 3. combine
  prefill_combine_kernel<T><<<p.B * p.T * p.Hq, D, 0, s>>>(p, PrefillCfg<D>::C);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && launches) *launches += 3;
  return e;
}

}  // namespace

int prefill_chunk_keys(int D) { return D == 64 ? PrefillCfg<64>::C : PrefillCfg<128>::C; }

bool prefill_supported(int dtype, int D, int G) {
  return (dtype == DKV_BF16 || dtype == DKV_FP16) && (D == 64 || D == 128) &&
         (G == 1 || G == 2 || G == 4 || G == 8);
}

cudaError_t launch_prefill(const PrefillParams& p, int dtype, cudaStream_t s, int* launches,
                           const void* wq, const KernelTimer& timer) {
  const int G = p.Hq / p.Hkv;
#define DKV_P(TT, DD, GG) \
  if (p.D == DD && G == GG) return launch_prefill_t<TT, DD, GG>(p, s, launches, wq, timer);
  if (dtype == DKV_BF16) {
    DKV_P(__nv_bfloat16, 64, 1) DKV_P(__nv_bfloat16, 64, 2) DKV_P(__nv_bfloat16, 64, 4)
    DKV_P(__nv_bfloat16, 64, 8) DKV_P(__nv_bfloat16, 128, 1) DKV_P(__nv_bfloat16, 128, 2)
    DKV_P(__nv_bfloat16, 128, 4) DKV_P(__nv_bfloat16, 128, 8)
  } else {
    DKV_P(__half, 64, 1) DKV_P(__half, 64, 2) DKV_P(__half, 64, 4) DKV_P(__half, 64, 8)
    DKV_P(__half, 128, 1) DKV_P(__half, 128, 2) DKV_P(__half, 128, 4) DKV_P(__half, 128, 8)
  }
#undef DKV_P
  return cudaErrorInvalidValue;
}

}  // namespace dkv
