// tc_dq.cu -- gradients of the orthogonal blocks, summed over tokens, on the tensor cores.
//
// Backward of the block-diagonal applies of "POET-X: Memory-efficient LLM
// Training by Scaling Orthogonal Transformation" (gist.science summary,
// sections 2.C and 2.E -- the page only says "autograd"; this is the plain
// chain rule): for every block j
//     dQ_j[i][k] = sum_t G[t][j*b + i] * V[t][j*b + k]
// where both operands are token-major activations whose block j occupies the
// contiguous columns [j*b, j*b + b):
//   R side  G = dy gathered by perm_out, V = z             (dQ_R)
//   P side  G = g_u,                     V = x gathered by perm_in   (dQ_P)
// (the gathers are made once, in one pass over HBM, by tc_permute.cu).
// The contraction runs over tokens: tcgen05.mma with M = 128 rows i, N = b
// columns k, K = 16 tokens, both operands MN-major tiles of [64 tokens x b
// features] brought in by TMA (128-byte swizzle) through a multi-stage ring.
// A CTA owns one block and a contiguous range of 64-token chunks; its fp32
// accumulator lives in TMEM and is written, at the end, to the CTA's own slot
// of a partial-sum buffer [splits][d][b]; the consumer adds the slots in a
// fixed order, so the result does not depend on scheduling.  All waits are
// bounded.
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

constexpr int kThreads = 192;        // warp 0: TMA; warp 1: MMA; warps 2..5: epilogue
constexpr int KT = 64;               // tokens per pipeline stage
constexpr int kSmemMax = 232448;
constexpr int kMaxStages = 8;
constexpr int kMaxSplit = 9;

template <int B>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmV,
              int nb, int n_chunks, int n_split, int stages, float* __restrict__ part, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int tile_bytes = KT * B * 2;
  constexpr int halves = B / 128;
  constexpr uint32_t ncols = halves * B;
  uint8_t* tiles = smem;   // per stage: [G tile][V tile]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + stages * 2 * tile_bytes);
  uint64_t* empty = full + kMaxStages;
  uint64_t* dfull = empty + kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dfull + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int j = blockIdx.x % nb;
  const int split = blockIdx.x / nb;
  const int c_begin = (int)((long long)split * n_chunks / n_split);
  const int c_end = (int)((long long)(split + 1) * n_chunks / n_split);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(full + s, 1);
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
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      for (int c = c_begin; c < c_end && ok; ++c) {
        if (!(ok = mbar_wait(empty + st, ph ^ 1, err))) break;
        mbar_arrive_expect_tx(full + st, 2 * tile_bytes);
        uint8_t* dst = tiles + st * 2 * tile_bytes;
#pragma unroll
        for (int q = 0; q < B / 64; ++q) {
          tma_load_2d(dst + q * (KT * 128), &tmG, j * B + q * 64, c * KT, full + st);
          tma_load_2d(dst + tile_bytes + q * (KT * 128), &tmV, j * B + q * 64, c * KT, full + st);
        }
        if (++st == stages) { st = 0; ph ^= 1; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, B, true, true);
      int st = 0;
      uint32_t ph = 0;
      for (int c = c_begin; c < c_end && ok; ++c) {
        if (!(ok = mbar_wait(full + st, ph, err))) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(tiles + st * 2 * tile_bytes);
        const uint32_t b_base = a_base + tile_bytes;
#pragma unroll
        for (int h = 0; h < halves; ++h) {
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk) {
            // A: features [h*128, h*128+128) of the G tile; B: all b features of the V tile
            const uint64_t adesc = sw128_desc(a_base + h * 2 * (KT * 128) + kk * 2048, KT * 128, 1024);
            const uint64_t bdesc = sw128_desc(b_base + kk * 2048, KT * 128, 1024);
            mma_bf16(tmem_base + (uint32_t)(h * B), adesc, bdesc, idesc, (c != c_begin || kk) ? 1u : 0u);
          }
        }
        mma_commit(empty + st);
        if (++st == stages) { st = 0; ph ^= 1; }
      }
      mma_commit(dfull);
    }
  } else {
    // epilogue warps 2..5 own TMEM lane quarters (warp % 4): rows i, columns k
    const int quarter = warp % 4;
    const bool any = c_end > c_begin;
    if (any && mbar_wait(dfull, 0, err)) tc_fence_after();
    float* slot = part + (size_t)split * nb * B * B;
    for (int h = 0; h < halves; ++h) {
      const int i = h * 128 + quarter * 32 + lane;
      float4* drow = reinterpret_cast<float4*>(slot + ((size_t)j * B + i) * B);
      for (int c0 = 0; c0 < B; c0 += 32) {
        uint32_t r[32];
        if (any) {
          tmem_ld32(tmem_base + (uint32_t)(h * B + c0) + ((uint32_t)(quarter * 32) << 16), r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int v = 0; v < 32; ++v) r[v] = 0u;   // an empty token range contributes zero
        }
#pragma unroll
        for (int v = 0; v < 32; v += 4)
          drow[(c0 + v) / 4] = make_float4(__uint_as_float(r[v]), __uint_as_float(r[v + 1]),
                                           __uint_as_float(r[v + 2]), __uint_as_float(r[v + 3]));
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

// Token splits per block: enough CTAs to keep HBM busy, few enough that the
// partial sums (b x b fp32 per CTA) stay a small part of the traffic.
int dq_splits(int T, int d, int b) {
  const int sms = device_sm_count();
  const int nb = d / b;
  const int n_chunks = (T + KT - 1) / KT;
  int n_split = sms / nb;
  if (n_split > kMaxSplit) n_split = kMaxSplit;
  if (n_split > n_chunks) n_split = n_chunks;
  if (n_split < 1) n_split = 1;
  return n_split;
}

// part[s][j][i][k] = sum over split s's tokens of G[t][jb+i] V[t][jb+k], s < n_split.
poetx_status dq_bf16(const void* G, const void* V, int T, int d, int b, int n_split, float* part,
                     cudaStream_t s) {
  if (!dq_supported(d, b) || n_split < 1 || n_split > kMaxSplit) return POETX_ERR_UNSUPPORTED;
  if (T <= 0) {
    if (cudaMemsetAsync(part, 0, sizeof(float) * (size_t)n_split * d * b, s) != cudaSuccess)
      return check_launch();
    return POETX_OK;
  }
  CUtensorMap tg, tv;
  if (!make_tmap_2d(&tg, G, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d, KT, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tv, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d, KT, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return POETX_ERR_CUDA;
  const int nb = d / b;
  const int n_chunks = (T + KT - 1) / KT;
  const int tile_bytes = KT * b * 2;
  int stages = (kSmemMax - 1024 - 256) / (2 * tile_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  const int smem = stages * 2 * tile_bytes + 1024 + 256;
  int* err = device_error_word();
  auto kern = b == 256 ? dq_kernel<256> : dq_kernel<128>;
  set_max_dynamic_smem((const void*)kern, smem);
  {
    KernelScope ks_("tc_dq", s);
    kern<<<nb * n_split, kThreads, smem, s>>>(tg, tv, nb, n_chunks, n_split, stages, part, err);
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
