// tc_gemm.cu -- the frozen-weight products on the 5th-generation tensor cores.
//
// [POET-X §2.A] ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", gist.science summary, section 2.A): the layer is applied
// to the activations; the only dense product is the one with the frozen,
// permutation-merged weight W0m:
//   forward   z   = u   . W0m^T   (B = W0m [N = d_out, K = d_in], K-major)
//   backward  g_u = g_z . W0m     (B = W0m [K = d_out, N = d_in], MN-major)
// C[M, N] (bf16) = A[M, K] (bf16, K-major) . B^T, fp32 accumulation in TMEM.
//
// Persistent kernel on CTA pairs (clusters of two): one pair computes a
// 256 x 256 output tile with 64-deep k steps.  Each CTA of the pair loads 128
// rows of A and 128 columns of B per k step (32 KB) into its own 6-stage
// shared-memory ring; the pair's first CTA issues tcgen05.mma.cta_group::2
// (M = 256, N = 256, K = 16), which reads both CTAs' shared memory and writes
// each CTA's 128 accumulator rows into that CTA's tensor memory.  Per SM the
// operand traffic is 32 KB per k step instead of the 48 KB of a one-CTA
// 128 x 256 tile, for the same MMA work.  Tiles go out column block fastest,
// so the pairs of one round share a few row blocks of A while they are in L2.
//   warp 0     one thread per CTA issues that CTA's TMA loads; their bytes
//              are counted on the first CTA's `full` barrier;
//   warp 1     allocates 512 TMEM columns in both CTAs (two 256-column
//              accumulators); in the first CTA one thread issues the MMAs and
//              frees each stage in both CTAs with a multicast commit;
//   warps 2-5  drain an accumulator (tcgen05.ld), round to bf16 and store,
//              while the MMAs fill the other one; both CTAs' drains are
//              counted on the first CTA's `tempty` barrier.
// Every wait is bounded (see tc_ptx.cuh); on expiry the kernel records
// POETX_ERR_TIMEOUT in the library's error word and winds down (the first
// CTA waits, bounded, for the loads and MMAs already issued before the pair
// frees its tensor memory).
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

constexpr int BM = 256, BN = 256, BK = 64, STAGES = 6;
constexpr int HM = BM / 2, HN = BN / 2;   // rows of A / columns of B in each CTA
constexpr int A_BYTES = HM * BK * 2;      // 16 KB
constexpr int B_BYTES = HN * BK * 2;      // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDrainLimit = 1u << 16;   // bounded waits of the wind-down after an error

__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB, __nv_bfloat16* __restrict__ C,
                          int M, int N, int K, int b_mn, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();   // 0: the pair's first CTA (issues the MMAs)
  const int pair = blockIdx.x / 2, n_pairs = gridDim.x / 2;
  const int m_tiles = (M + BM - 1) / BM, n_tiles = N / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int k_iters = K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, 2 * 128);   // both CTAs' epilogue threads
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // this CTA's halves of every stage; bytes counted on the first CTA's `full`
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int issued = 0;
      for (int tile = pair; tile < num_tiles && ok; tile += n_pairs) {
        const int m_blk = tile / n_tiles, n_blk = tile % n_tiles;
        const int row0 = m_blk * BM + (int)rank * HM;
        const int col0 = n_blk * BN + (int)rank * HN;
        for (int kb = 0; kb < k_iters; ++kb) {
          if (!(ok = mbar_wait(empty + stage, phase ^ 1, err))) break;
          if (rank == 0) mbar_arrive_expect_tx(full + stage, 2 * STAGE_BYTES);
          const uint32_t fb = mapa_shared(smem_u32(full + stage), 0);
          tma_load_2d_pair(sA + stage * A_BYTES, &tmA, kb * BK, row0, fb);
          if (!b_mn) {
            tma_load_2d_pair(sB + stage * B_BYTES, &tmB, kb * BK, col0, fb);
          } else {
#pragma unroll
            for (int q = 0; q < HN / 64; ++q)
              tma_load_2d_pair(sB + stage * B_BYTES + q * (BK * 128), &tmB, col0 + q * 64,
                               kb * BK, fb);
          }
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok && rank == 0) {
        // wind-down: the loads already issued land before the pair exits
        // (the last `issued` stages; `full` counts both CTAs' bytes)
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < STAGES && i < issued; ++i) {
          if (--s < 0) { s = STAGES - 1; ph ^= 1; }
          mbar_wait_bounded(full + s, ph, kDrainLimit, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, BN, false, b_mn != 0);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += n_pairs) {
        if (!(ok = mbar_wait_cluster(tempty + acc, acc_phase ^ 1, err))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < k_iters; ++kb) {
          if (!(ok = mbar_wait(full + stage, phase, err))) break;
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t adesc = sw128_desc(a_base + k * 32, 16, 1024);
            const uint64_t bdesc = b_mn ? sw128_desc(b_base + k * 2048, BK * 128, 1024)
                                        : sw128_desc(b_base + k * 32, 16, 1024);
            mma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb | k) != 0);
          }
          mma_commit_pair(empty + stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit_pair(tfull + acc);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      // every MMA issued has finished before the tensor memory is freed
      mma_commit_pair_local(mma_done);
      mbar_wait_bounded(mma_done, 0, ok ? kWaitLimit : kDrainLimit, ok ? err : nullptr);
    }
  } else {
    // epilogue warps 2..5 own TMEM lane quarters (warp % 4)
    const int quarter = warp % 4;
    const int row_in_tile = (int)rank * HM + quarter * 32 + lane;
    const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < num_tiles; tile += n_pairs) {
      const int m_blk = tile / n_tiles, n_blk = tile % n_tiles;
      // one thread waits, the other epilogue threads sleep at a named barrier
      bool lok = true;
      if (quarter == 2 && lane == 0) lok = mbar_wait(tfull + acc, acc_phase, err);
      if (bar_sync_or(1, 128, !lok)) break;
      tc_fence_after();
      const int row = m_blk * BM + row_in_tile;
      __nv_bfloat16* crow = C + (size_t)row * N + (size_t)n_blk * BN;
      const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        tmem_ld32(tbase + c, r);
        tmem_ld_wait();
        tmem_regs_ready(r);
        if (row < M) {
          uint4* dst = reinterpret_cast<uint4*>(crow + c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
            o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
            o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
            o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
            dst[v] = o;
          }
        }
      }
      tc_fence_before();
      // the accumulator may be refilled once both CTAs have drained it
      mbar_arrive_remote(tempty0 + (uint32_t)(acc * 8));
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no CTA frees its tensor memory or leaves while the pair still works
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

bool gemm_supported(int N, int K) { return N % BN == 0 && K % BK == 0 && N > 0 && K > 0; }

// C[M,N] = A[M,K] . B^T; B is [N,K] (b_mn == false) or [K,N] (b_mn == true), all bf16 row-major.
poetx_status gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, bool b_mn,
                       cudaStream_t s, int reserve_sms) {
  if (M <= 0) return POETX_OK;
  if (!gemm_supported(N, K)) return POETX_ERR_UNSUPPORTED;
  CUtensorMap ta, tb;
  if (!make_tmap_2d(&ta, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)M, (uint64_t)K, HM, BK,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return POETX_ERR_CUDA;
  const bool okb =
      b_mn ? make_tmap_2d(&tb, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)K, (uint64_t)N, BK,
                          64, CU_TENSOR_MAP_SWIZZLE_128B)
           : make_tmap_2d(&tb, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)N, (uint64_t)K, HN,
                          BK, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!okb) return POETX_ERR_CUDA;
  // as few pairs as give the fewest rounds of tiles (the SMs left over stay
  // free for work on another stream); the reserved SMs stay out of the grid
  // unless leaving them out would add a round
  const int tiles = ((M + BM - 1) / BM) * (N / BN);
  const int all_pairs = device_sm_count() / 2 > 0 ? device_sm_count() / 2 : 1;
  const int min_rounds = (tiles + all_pairs - 1) / all_pairs;
  int avail = (device_sm_count() - (reserve_sms > 0 ? reserve_sms : 0)) / 2;
  if (avail < 1) avail = 1;
  int rounds = (tiles + avail - 1) / avail;
  if (rounds > min_rounds) rounds = min_rounds;
  const int pairs = (tiles + rounds - 1) / rounds;
  if (set_max_dynamic_smem((const void*)gemm_bf16_pair_kernel, SMEM_BYTES) != cudaSuccess)
    return check_launch();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    KernelScope ks_(b_mn ? "tc_gemm_nn" : "tc_gemm_nt", s);
    if (cudaLaunchKernelEx(&cfg, gemm_bf16_pair_kernel, ta, tb, (__nv_bfloat16*)C, M, N, K,
                           b_mn ? 1 : 0, device_error_word()) != cudaSuccess)
      return check_launch();
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
