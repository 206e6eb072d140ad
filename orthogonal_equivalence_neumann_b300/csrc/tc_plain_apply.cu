// tc_plain_apply.cu -- block-diagonal apply of contiguous block columns, Q resident in tensor memory.
//
// [POET-X §2.C] ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", gist.science summary, section 2.C): the orthogonal factors
// are block-diagonal, each b x b block its own small matrix, processed as a
// batch.  This kernel computes, for every token t and block j,
//     out[t][j*b + i] = sum_k Qop_j[i][k] in[t][j*b + k],   Qop_j = Q_j or Q_j^T,
// with the block's columns contiguous in both tensors (no permutation).  It
// serves the layers whose permuted applies do not fit the cluster exchange
// (tc_cluster_apply.cu): there the permutation runs as a separate column
// gather (tc_permute.cu) before a gathered apply, or after a scattered one
// (the inverse permutation gathers the block outputs into place).
//
// One CTA per (block j, token stripe): it keeps Qop_j in tensor memory for
// the whole launch (tc_qstage.cuh) and walks the 128-token tiles r, r + R,
// r + 2R, ... of its stripe r:
//   warp 0      TMA: the tile's block columns [128 tokens x b] (128-byte
//               swizzle, K-major: the MMA's B operand as loaded)
//   warp 1      MMA (lane 0): M = 128 outputs per half of the block, N = 128
//               tokens, K = 16, A from TMEM, each half into its own 128-column
//               accumulator slot (b = 256: one slot per half, handed to the
//               epilogue and back half by half; b = 128: two slots in turn)
//   warps 2..9  epilogue, two warps per TMEM lane quarter (each drains 64 of
//               the tile's tokens): TMEM -> bf16 token rows in the slot's
//               staging tile (the TMA store layout) -> TMA store, so one half's
//               store overlaps the next half's drain
// Every wait is bounded (tc_ptx.cuh).
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"
#include "tc_qstage.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

constexpr int kPaEpiWarps = 8;
constexpr int kPaEpiThreads = 32 * kPaEpiWarps;
constexpr int kPaThreads = 64 + kPaEpiThreads;
constexpr int kPaTT = 128;             // tokens per tile: the MMA's N
constexpr int kPaSlots = 2;            // 128-column accumulator slots = staging tiles
constexpr int kPaStg = kPaTT * 128 * 2;   // one staging tile: 128 tokens x 128 features bf16
constexpr int kPaMaxNS = 8;

struct PaGeo {
  int NS;          // input stages
  int s_bytes;     // one input tile: 128 tokens x b bf16
  int q_cols, tmem_cols;
  int smem;
};

// Shared memory: 1 KB of barriers, NS input stages, two staging tiles.  Q is
// staged in the stages and staging tiles (contiguous) before the first tile
// loads, which needs NS * s_bytes + 2 * kPaStg >= b * b * 2.
bool pa_geometry(int b, PaGeo* g) {
  if (b != 128 && b != 256) return false;
  g->s_bytes = kPaTT * b * 2;
  g->NS = 0;
  for (int ns = kPaMaxNS; ns >= 2; --ns)
    if (1024 + 1024 + ns * g->s_bytes + kPaSlots * kPaStg <= 232448 &&
        ns * g->s_bytes + kPaSlots * kPaStg >= b * b * 2) {
      g->NS = ns;
      break;
    }
  if (g->NS == 0) return false;
  g->q_cols = (b / 128) * (b / 2);
  const int used = g->q_cols + kPaSlots * kPaTT;
  g->tmem_cols = 32;
  while (g->tmem_cols < used) g->tmem_cols *= 2;
  g->smem = 1024 + 1024 + g->NS * g->s_bytes + kPaSlots * kPaStg;
  return g->tmem_cols <= 512;
}

__device__ __forceinline__ void pa_epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kPaEpiThreads) : "memory");
}

// Accumulator slot (= staging tile) of half h of the it-th tile, and how many
// times the slot was used before.
template <int B>
__device__ __forceinline__ int pa_slot(int it, int h) { return B == 256 ? h : (it & 1); }
template <int B>
__device__ __forceinline__ int pa_use(int it) { return B == 256 ? it : (it >> 1); }

template <int B>
__global__ void __launch_bounds__(kPaThreads, 1)
    pa_kernel(const __grid_constant__ CUtensorMap tmIn, const __grid_constant__ CUtensorMap tmOut,
              const __grid_constant__ CUtensorMap tmQ, int T, int nb, PaGeo g, int transpose_q,
              int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int halves = B / 128;
  constexpr int TT = kPaTT;
  uint64_t* s_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* s_empty = s_full + kPaMaxNS;
  uint64_t* a_full = s_empty + kPaMaxNS;    // per accumulator slot
  uint64_t* a_empty = a_full + kPaSlots;
  uint64_t* q_full = a_empty + kPaSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 1);
  uint8_t* sbuf = smem + 1024;
  uint8_t* obuf = sbuf + g.NS * g.s_bytes;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int j = (int)blockIdx.x % nb;
  const int stripe = (int)blockIdx.x / nb;
  const int stripes = (int)gridDim.x / nb;
  const int n_tiles = (T + TT - 1) / TT;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPaMaxNS; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(s_empty + i, 1);
    }
    for (int i = 0; i < kPaSlots; ++i) {
      mbar_init(a_full + i, 1);
      mbar_init(a_empty + i, kPaEpiThreads);
    }
    mbar_init(q_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, (uint32_t)g.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  bool ok = true;
  // Qop_j into tensor memory through the stages and staging tiles, before any tile loads
  if (threadIdx.x == 0) issue_q_loads(&tmQ, sbuf, j, 1, B, q_full);
  if (warp >= 2 && warp < 6) {
    if ((ok = mbar_wait(q_full, 0, err))) q_stage_to_tmem<B>(sbuf, 1, transpose_q, tmem_base, warp % 4, lane);
  }
  tc_fence_before();
  fence_proxy_async_smem();   // the staging reads are done before TMA overwrites the stages
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  tc_fence_after();

  const uint32_t acc0 = tmem_base + (uint32_t)g.q_cols;
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      for (int it = 0, tile = stripe; tile < n_tiles && ok; tile += stripes, ++it) {
        const int s = it % g.NS;
        if (!(ok = mbar_wait(s_empty + s, ((it / g.NS) & 1) ^ 1, err))) break;
        mbar_arrive_expect_tx(s_full + s, (uint32_t)g.s_bytes);
        uint8_t* dst = sbuf + s * g.s_bytes;
        for (int q = 0; q < B / 64; ++q)
          tma_load_2d(dst + q * (TT * 128), &tmIn, j * B + q * 64, tile * TT, s_full + s);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, TT, false, false);
      for (int it = 0, tile = stripe; tile < n_tiles && ok; tile += stripes, ++it) {
        const int s = it % g.NS;
        if (!(ok = mbar_wait(s_full + s, (it / g.NS) & 1, err))) break;
        const uint32_t sb = smem_u32(sbuf + s * g.s_bytes);
        for (int h = 0; h < halves && ok; ++h) {
          const int slot = pa_slot<B>(it, h);
          if (!(ok = mbar_wait(a_empty + slot, (pa_use<B>(it) & 1) ^ 1, err))) break;
          tc_fence_after();
          const uint32_t d_tmem = acc0 + (uint32_t)(slot * TT);
          const uint32_t a_tmem = tmem_base + (uint32_t)(h * (B / 2));
#pragma unroll 4
          for (int kk = 0; kk < B / 16; ++kk) {
            const uint64_t bdesc = sw128_desc(sb + (kk >> 2) * (TT * 128) + (kk & 3) * 32, 16, 1024);
            mma_bf16_ts(d_tmem, a_tmem + (uint32_t)(kk * 8), bdesc, idesc, kk != 0);
          }
          mma_commit(a_full + slot);
        }
        mma_commit(s_empty + s);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    // TMEM lanes are output features, columns tokens: each thread writes its
    // feature's 64 tokens into the slot's token-row staging tile (128-byte
    // swizzle, the TMA store layout); one thread then stores it with TMA.
    const int quarter = warp % 4;
    const int et = threadIdx.x - 64;   // 0 .. kPaEpiThreads - 1
    const int part = (warp - 2) / 4;   // tokens [64 part, +64) of the tile
    const int f = quarter * 32 + lane; // output feature within the half
    bool any = false;
    for (int it = 0, tile = stripe; tile < n_tiles && ok; tile += stripes, ++it) {
      for (int h = 0; h < halves; ++h) {
        const int slot = pa_slot<B>(it, h), use = pa_use<B>(it);
        uint8_t* ostg = obuf + slot * kPaStg;
        if (!(ok = mbar_wait(a_full + slot, use & 1, err))) break;
        tc_fence_after();
        if (use > 0) {   // the store that last used this staging tile has read it
          if (et == 0)
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          pa_epi_bar();
        }
        uint8_t* col = ostg + (f >> 6) * (TT * 128) + (f & 7) * 2;
        const uint32_t fu = (uint32_t)((f & 63) >> 3);
        const uint32_t tacc = acc0 + (uint32_t)(slot * TT + part * 64) + ((uint32_t)(quarter * 32) << 16);
        uint32_t rr[2][32];
        tmem_ld32(tacc, rr[0]);
        tmem_ld32(tacc + 32u, rr[1]);
        tmem_ld_wait();
        tmem_regs_ready(rr[0]);
        tmem_regs_ready(rr[1]);
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const int tr = part * 64 + e;
          *reinterpret_cast<__nv_bfloat16*>(col + tr * 128 + ((fu ^ (uint32_t)(tr & 7)) << 4)) =
              __float2bfloat16_rn(__uint_as_float(rr[e >> 5][e & 31]));
        }
        tc_fence_before();
        mbar_arrive(a_empty + slot);   // the slot may be refilled
        fence_proxy_async_smem();
        pa_epi_bar();
        if (et == 0) {
          for (int q = 0; q < 2; ++q)
            tma_store_2d(&tmOut, ostg + q * (TT * 128), j * B + h * 128 + q * 64, tile * TT);
          bulk_commit();
        }
        any = true;
      }
    }
    if (et == 0 && any) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)g.tmem_cols);
  }
}

}  // namespace

bool plain_apply_supported(int d, int b) {
  PaGeo g;
  return d > 0 && d % b == 0 && d / b <= 65535 && pa_geometry(b, &g);
}

poetx_status plain_apply_bf16(const void* in, void* out, const void* Q, int T, int d, int b,
                              bool transpose_q, cudaStream_t s) {
  if (T <= 0) return POETX_OK;
  PaGeo g;
  if (!plain_apply_supported(d, b) || !pa_geometry(b, &g)) return POETX_ERR_UNSUPPORTED;
  const int nb = d / b;
  const int n_tiles = (T + kPaTT - 1) / kPaTT;
  int stripes = device_sm_count() / nb;
  if (stripes < 1) stripes = 1;
  if (stripes > n_tiles) stripes = n_tiles;
  if ((long long)stripes * nb > 2147483647LL) return POETX_ERR_SHAPE;
  CUtensorMap tin, tout, tq;
  if (!make_tmap_2d(&tin, in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d, kPaTT, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tout, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d, kPaTT, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d, (uint64_t)b, 64, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return POETX_ERR_CUDA;
  const void* kern = b == 256 ? (const void*)pa_kernel<256> : (const void*)pa_kernel<128>;
  if (set_max_dynamic_smem(kern, g.smem) != cudaSuccess) return check_launch();
  int* err = device_error_word();
  const int tqf = transpose_q ? 1 : 0;
  {
    KernelScope ks_("tc_plain_apply", s);
    if (b == 256)
      pa_kernel<256><<<stripes * nb, kPaThreads, g.smem, s>>>(tin, tout, tq, T, nb, g, tqf, err);
    else
      pa_kernel<128><<<stripes * nb, kPaThreads, g.smem, s>>>(tin, tout, tq, T, nb, g, tqf, err);
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
