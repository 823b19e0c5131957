// Projection GEMM on the 5th-generation tensor cores: Y[M,N] = X[M,K] . W[K,N]
// (the Q projection of a prefill, q = x.Wq, "Paper Notes: DirectKV",
// Fundamental Underlying Technologies, Kernel Fusion).
//
// One CTA computes a 128 x 128 tile of Y.  TMA streams 64-wide K blocks of X
// (K-major, 128-byte swizzle) and of W (N contiguous, i.e. MN-major, 128-byte
// swizzle) into a 3-stage shared-memory ring; one thread issues
// tcgen05.mma (M=128, N=128, K=16) into a TMEM accumulator; after the last
// block the four warps read the accumulator back (one TMEM lane per thread),
// round to the storage dtype and store.  Two CTAs fit on an SM, so one CTA's
// epilogue overlaps the other's main loop.
#include <mutex>

#include "tc_common.cuh"

namespace dkv {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 64, kStages = 3;
constexpr int kThreads = 128;
constexpr int kABytes = kBM * kBK * 2;        // 16 KB
constexpr int kBBytes = kBK * kBN * 2;        // 16 KB (two 64-column blocks)
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmem = 1024 /*align slack*/ + kStages * kStageBytes + 256;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   T* __restrict__ y, int M, int N, int K, DeviceStatus* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_s + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const int nk = (K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc::prefetch_tmap(&map_a);
    tc::prefetch_tmap(&map_b);
  }
  if (warp == 2) tc::tmem_alloc(tmem_base_s, kBN);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_base_s;

  if (threadIdx.x == 0) {
    // ---- TMA producer
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait_bounded(&empty[s], ((kb / kStages) & 1) ^ 1, abort_flag)) {
        record_timeout(status, kSiteEmpty);
        *abort_flag = 1;
        break;
      }
      uint8_t* a_s = ring + s * kStageBytes;
      uint8_t* b_s = a_s + kABytes;
      tc::mbar_expect_tx(&full[s], kStageBytes);
      tc::tma_load_2d(a_s, &map_a, kb * kBK, m0, &full[s]);
      tc::tma_load_2d(b_s, &map_b, n0, kb * kBK, &full[s]);
      tc::tma_load_2d(b_s + kBBytes / 2, &map_b, n0 + 64, kb * kBK, &full[s]);
    }
  } else if (threadIdx.x == 32) {
    // ---- MMA issuer
    constexpr uint32_t idesc_bf = tc::idesc_f16(true, kBM, kBN, false, true);
    constexpr uint32_t idesc_h = tc::idesc_f16(false, kBM, kBN, false, true);
    const uint32_t idesc = DT<T>::code == DKV_BF16 ? idesc_bf : idesc_h;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait_bounded(&full[s], (kb / kStages) & 1, abort_flag)) {
        record_timeout(status, kSiteFull);
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      const uint32_t a_addr = smem_u32(ring + s * kStageBytes);
      const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t ad = tc::sdesc_sw128(a_addr + kk * 32, 16, 1024);
        const uint64_t bd = tc::sdesc_sw128(b_addr + kk * 16 * 128, kBBytes / 2, 1024);
        tc::mma_ss(tmem, ad, bd, idesc, (kb | kk) != 0);
      }
      tc::mma_commit(&empty[s]);
    }
    tc::mma_commit(acc_full);
  }

  // ---- epilogue: all four warps, one accumulator row per thread
  __syncwarp();
  bool ok = mbar_wait_bounded(acc_full, 0, abort_flag);
  ok = __all_sync(0xffffffffu, ok && !*abort_flag);  // tcgen05.ld needs the whole warp
  tc::fence_after_sync();
  const int row = warp * 32 + lane;
  const int gm = m0 + row;
  if (ok) {
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      uint32_t r[32];
      tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, r);
      tc::tmem_wait_ld();
      const int gn = n0 + c * 32;
      if (gm < M && gn < N) {
        uint4* dst = reinterpret_cast<uint4*>(y + (size_t)gm * N + gn);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 o;
          o.x = tc::pack2<T>(__uint_as_float(r[v * 8 + 0]), __uint_as_float(r[v * 8 + 1]));
          o.y = tc::pack2<T>(__uint_as_float(r[v * 8 + 2]), __uint_as_float(r[v * 8 + 3]));
          o.z = tc::pack2<T>(__uint_as_float(r[v * 8 + 4]), __uint_as_float(r[v * 8 + 5]));
          o.w = tc::pack2<T>(__uint_as_float(r[v * 8 + 6]), __uint_as_float(r[v * 8 + 7]));
          if (gn + v * 8 < N) dst[v] = o;
        }
      }
    }
  } else if (lane == 0) {
    record_timeout(status, kSiteFull);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) tc::tmem_dealloc(tmem, kBN);
}

// ---- host: tensor maps ---------------------------------------------------------
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

}  // namespace

// Row-major [rows, cols] matrix of 16-bit elements; box = box_cols x box_rows,
// 128-byte swizzle (box_cols * 2 must be 128).
bool make_tmap_2d(CUtensorMap* map, const void* base, int dtype, uint64_t rows, uint64_t cols,
                  uint32_t box_cols, uint32_t box_rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype == DKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same without swizzle: a box lands as box_rows dense rows of box_cols * 2
// bytes (the decode projection's 32-column weight blocks and x's columns).
bool make_tmap_2d_plain(CUtensorMap* map, const void* base, int dtype, uint64_t rows,
                        uint64_t cols, uint32_t box_cols, uint32_t box_rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype == DKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Q as [tokens][Hq][D] (row-major [tokens, Hq*D]); box = 64 of D x G heads x
// TQ tokens, so a box lands as G*TQ rows of 128 bytes, ordered (token, head).
bool make_tmap_q(CUtensorMap* map, const void* q, int dtype, int D, int Hq, uint64_t tokens,
                 int G, int TQ) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, tokens};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)TQ};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype == DKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  3, const_cast<void*>(q), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp16 partials [blocks][rows][D]: box = 64 of D x 128 rows x 1 block.
bool make_tmap_partial(CUtensorMap* map, void* base, int D, uint64_t rows, uint64_t blocks) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, rows, blocks};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, rows * D * 2};
  cuuint32_t box[3] = {64, 32, 1};  // one warp's 32 rows
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_gemm_tc(const void* x, const void* w, void* y, int M, int N, int K, int dtype,
                           DeviceStatus* status, cudaStream_t s) {
  if (M <= 0 || N <= 0 || K <= 0 || N % 64 != 0 || K % 8 != 0) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  if (!make_tmap_2d(&ma, x, dtype, M, K, kBK, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&mb, w, dtype, K, N, 64, kBK)) return cudaErrorInvalidValue;
  dim3 grid((N + kBN - 1) / kBN, (M + kBM - 1) / kBM);
  if (dtype == DKV_BF16) {
    auto k = gemm_tc_kernel<__nv_bfloat16>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    k<<<grid, kThreads, kSmem, s>>>(ma, mb, static_cast<__nv_bfloat16*>(y), M, N, K, status);
  } else {
    auto k = gemm_tc_kernel<__half>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    k<<<grid, kThreads, kSmem, s>>>(ma, mb, static_cast<__half*>(y), M, N, K, status);
  }
  return cudaGetLastError();
}

}  // namespace dkv
