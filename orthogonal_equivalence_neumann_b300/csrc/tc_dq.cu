// tc_dq.cu -- gradients of the orthogonal blocks, summed over tokens, on the tensor cores.
//
// Backward of the block-diagonal applies of "POET-X: Memory-efficient LLM
// Training by Scaling Orthogonal Transformation" (gist.science summary,
// sections 2.C and 2.E -- the page only says "autograd"; this is the plain
// chain rule): for every block j
//     dQ_j[i][k] = sum_t G[t][gG(j*b + i)] * V[t][gV(j*b + k)]
// with exactly one of the two column maps a permutation (gather) and the
// other the identity:
//   R side  G = dy gathered by perm_out, V = z      (dQ_R)
//   P side  G = g_u,                     V = x gathered by perm_in   (dQ_P)
// The contraction runs over tokens: tcgen05.mma with M = 128 rows i, N = b
// columns k, K = 16 tokens, both operands MN-major tiles of [64 tokens x b
// features] with the 128-byte swizzle.  The identity-mapped operand arrives
// by TMA; the gathered one is assembled by 8 worker warps from global memory
// (the block's b columns of each token row).  A CTA owns one block and a
// token range (a multiple of 64 tokens); the fp32 accumulator lives in TMEM
// and is added to dQ (zeroed first) with vector reductions at the end.
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

constexpr int kThreads = 320;
constexpr int kWorkers = 256;
constexpr int KT = 64;               // tokens per pipeline stage
constexpr int kSmemMax = 232448;
constexpr int kMaxStages = 6;

__device__ __forceinline__ uint32_t sw128_offset(int r, int k, int rows) {
  return (uint32_t)((k >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// GATHER_A: the G operand (rows i) is gathered; otherwise V (columns k) is.
template <bool GATHER_A>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmId, const __nv_bfloat16* __restrict__ gsrc,
              const int32_t* __restrict__ perm, int T, int d, int b, int tok_per_cta,
              int stages, float* __restrict__ dQ, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int tile_bytes = KT * b * 2;
  uint8_t* tiles = smem;   // per stage: [A tile][B tile]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + stages * 2 * tile_bytes);
  uint64_t* full = bars;
  uint64_t* empty = full + kMaxStages;
  uint64_t* dfull = empty + kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dfull + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nb = d / b;
  const int j = blockIdx.x % nb;
  const int split = blockIdx.x / nb;
  const int tb = split * tok_per_cta;
  const int te = min(T, tb + tok_per_cta);
  const int chunks = tb < te ? (te - tb + KT - 1) / KT : 0;
  const int halves = b / 128;
  const uint32_t ncols = (uint32_t)(halves * b) < 32u ? 32u : (uint32_t)(halves * b);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(full + s, 1 + kWorkers);
      mbar_init(empty + s, 1);
    }
    mbar_init(dfull, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // operand placement within a stage: A (rows i, from G) first, then B (columns k, from V)
  const int id_off = GATHER_A ? tile_bytes : 0;   // the TMA-loaded operand
  const int ga_off = GATHER_A ? 0 : tile_bytes;   // the gathered operand

  if (warp == 0) {
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      for (int c = 0; c < chunks; ++c) {
        if (!mbar_wait(empty + st, ph ^ 1, err)) break;
        mbar_arrive_expect_tx(full + st, tile_bytes);
        uint8_t* dst = tiles + st * 2 * tile_bytes + id_off;
        for (int q = 0; q < b / 64; ++q)
          tma_load_2d(dst + q * (KT * 128), &tmId, j * b + q * 64, tb + c * KT, full + st);
        if (++st == stages) { st = 0; ph ^= 1; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, b, true, true);
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int c = 0; c < chunks && ok; ++c) {
        if (!(ok = mbar_wait(full + st, ph, err))) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(tiles + st * 2 * tile_bytes);
        const uint32_t b_base = a_base + tile_bytes;
        for (int h = 0; h < halves; ++h) {
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk) {
            // A: features [h*128, h*128+128) of the G tile; B: all b features of the V tile
            const uint64_t adesc = sw128_desc(a_base + h * 2 * (KT * 128) + kk * 2048, KT * 128, 1024);
            const uint64_t bdesc = sw128_desc(b_base + kk * 2048, KT * 128, 1024);
            mma_bf16(tmem_base + (uint32_t)(h * b), adesc, bdesc, idesc, (c | kk) != 0);
          }
        }
        mma_commit(empty + st);
        if (++st == stages) { st = 0; ph ^= 1; }
      }
      mma_commit(dfull);
    }
  } else {
    const int wt = threadIdx.x - 64;
    int st = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int c = 0; c < chunks && ok; ++c) {
      if (!(ok = mbar_wait(empty + st, ph ^ 1, err))) break;
      uint8_t* dst = tiles + st * 2 * tile_bytes + ga_off;
      const int t0 = tb + c * KT;
      // unit (t, f8): 8 consecutive gathered features of token t, one 16-byte store
      const int units = KT * (b / 8);
      for (int u = wt; u < units; u += kWorkers) {
        const int t = u / (b / 8), f8 = u % (b / 8);
        const int tt = t0 + t;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (tt < te) {
          const __nv_bfloat16* row = gsrc + (size_t)tt * d;
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const uint16_t v0 =
                __ldg(reinterpret_cast<const unsigned short*>(row + __ldg(perm + j * b + f8 * 8 + e)));
            const uint16_t v1 = __ldg(
                reinterpret_cast<const unsigned short*>(row + __ldg(perm + j * b + f8 * 8 + e + 1)));
            w[e / 2] = (uint32_t)v0 | ((uint32_t)v1 << 16);
          }
        }
        *reinterpret_cast<uint4*>(dst + sw128_offset(t, f8 * 8, KT)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(full + st);
      if (++st == stages) { st = 0; ph ^= 1; }
    }
    // epilogue: TMEM rows i (lanes), columns k -> atomically added to dQ_j
    if (ok && chunks > 0 && mbar_wait(dfull, 0, err)) {
      tc_fence_after();
      const int quarter = warp % 4;
      const int part = (warp - 2) / 4;          // 0 or 1
      for (int h = 0; h < halves; ++h) {
        const int i = h * 128 + quarter * 32 + lane;
        // the two warps of a lane quarter split the columns
        const int c_lo = part * (b / 2), c_hi = c_lo + b / 2;
        float* drow = dQ + ((size_t)j * b + i) * b;
        for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem_base + (uint32_t)(h * b + c0) + ((uint32_t)(quarter * 32) << 16), r);
          tmem_ld_wait();
#pragma unroll
          for (int v = 0; v < 32; v += 4)
            red_add_v4(drow + c0 + v, __uint_as_float(r[v]), __uint_as_float(r[v + 1]),
                       __uint_as_float(r[v + 2]), __uint_as_float(r[v + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, ncols);
  }
}

}  // namespace

bool dq_supported(int d, int b) { return (b == 128 || b == 256) && d % b == 0; }

poetx_status dq_bf16(const void* G, const void* V, int T, int d, int b, const int32_t* gG,
                     const int32_t* gV, float* dQ, cudaStream_t s) {
  if (cudaMemsetAsync(dQ, 0, sizeof(float) * (size_t)d * b, s) != cudaSuccess) return check_launch();
  if (T <= 0) return POETX_OK;
  if (!dq_supported(d, b) || (gG == nullptr) == (gV == nullptr)) return POETX_ERR_UNSUPPORTED;
  const bool gather_a = gG != nullptr;
  const void* id_src = gather_a ? V : G;
  const void* ga_src = gather_a ? G : V;
  const int32_t* perm = gather_a ? gG : gV;
  CUtensorMap tid;
  if (!make_tmap_2d(&tid, id_src, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d,
                    KT, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return POETX_ERR_CUDA;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int nb = d / b;
  int splits = sms / nb;
  if (splits < 1) splits = 1;
  int tok = (T + splits - 1) / splits;
  tok = (tok + KT - 1) / KT * KT;
  splits = (T + tok - 1) / tok;
  const int tile_bytes = KT * b * 2;
  int stages = (kSmemMax - 1024 - 256) / (2 * tile_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  const int smem = stages * 2 * tile_bytes + 1024 + 256;
  int* err = device_error_word();
  auto kern = gather_a ? dq_kernel<true> : dq_kernel<false>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  {
    KernelScope ks_(gather_a ? "tc_dq_gather_rows" : "tc_dq_gather_cols", s);
    kern<<<nb * splits, kThreads, smem, s>>>(tid, (const __nv_bfloat16*)ga_src, perm, T, d, b, tok,
                                             stages, dQ, err);
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
