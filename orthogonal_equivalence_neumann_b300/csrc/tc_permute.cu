// tc_permute.cu -- column permutation of token-major bf16 activations.
//
// [POET-X §2.B] ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", gist.science summary, section 2.B): permutations are index
// maps, applied by a gather, never as matrices:
//     out[t][c] = in[t][perm[c]]        (t < T, c < d)
// The backward's token sums of the block gradients read the gathered
// operands (dy gathered by perm_out, x gathered by perm_in) block by block;
// this kernel produces them in one pass over HBM (each element read and
// written once).
//
// Persistent CTAs walk slabs of TM whole token rows: one thread issues the
// TMA loads of a slab (128-byte swizzled boxes of TM x 64) into a two-slab
// ring, and eight worker warps build 16-byte output units (8 consecutive
// output columns of one token) from the swizzled slab and store them with
// coalesced writes.  All waits are bounded.
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

constexpr int kPermThreads = 288;   // warp 0: TMA; warps 1..8: workers
constexpr int kPermWorkers = 256;
constexpr int kPermSmemMax = 200 * 1024;

int permute_rows(int d) {
  for (int tm = 16; tm >= 8; tm /= 2)   // boxes start on 1024-byte swizzle atoms
    if (2 * tm * d * 2 <= kPermSmemMax) return tm;
  return 0;
}

__global__ void __launch_bounds__(kPermThreads, 1)
    permute_kernel(const __grid_constant__ CUtensorMap tmIn, __nv_bfloat16* __restrict__ out,
                   const int32_t* __restrict__ perm, int T, int d, int TM, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int slab_bytes = TM * d * 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + 2 * slab_bytes);
  uint64_t* empty = full + 2;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_slabs = (T + TM - 1) / TM;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kPermWorkers);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) {
      for (int it = 0, s = blockIdx.x; s < n_slabs; s += gridDim.x, ++it) {
        const int buf = it & 1;
        if (!mbar_wait(empty + buf, ((it >> 1) & 1) ^ 1, err)) break;
        mbar_arrive_expect_tx(full + buf, (uint32_t)slab_bytes);
        uint8_t* dst = smem + buf * slab_bytes;
        for (int c = 0; c < d / 64; ++c) tma_load_2d(dst + c * TM * 128, &tmIn, c * 64, s * TM, full + buf);
      }
    }
  } else {
    // a worker owns output column groups (8 columns); their 8 source columns
    // are fixed, so their slab offsets are computed once and reused for every
    // token of every slab
    const int wt = threadIdx.x - 32;
    const int groups = d / 8;
    constexpr int kMaxGroups = 4;   // d <= 8 * 256 * kMaxGroups
    uint32_t base[kMaxGroups][8], unit[kMaxGroups][8];
#pragma unroll
    for (int gi = 0; gi < kMaxGroups; ++gi) {
      const int c8 = (wt + gi * kPermWorkers) * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int a = c8 < d ? __ldg(perm + c8 + e) : 0;
        base[gi][e] = (uint32_t)((a >> 6) * TM * 128 + (a & 7) * 2);
        unit[gi][e] = (uint32_t)((a >> 3) & 7);
      }
    }
    for (int it = 0, s = blockIdx.x; s < n_slabs; s += gridDim.x, ++it) {
      const int buf = it & 1;
      if (!mbar_wait(full + buf, (it >> 1) & 1, err)) break;
      const uint8_t* slab = smem + buf * slab_bytes;
      const int t0 = s * TM;
      const int rows = min(TM, T - t0);
#pragma unroll
      for (int gi = 0; gi < kMaxGroups; ++gi) {
        const int g = wt + gi * kPermWorkers;
        if (g >= groups) break;
        for (int t = 0; t < rows; ++t) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const uint16_t va = *reinterpret_cast<const uint16_t*>(
                slab + base[gi][e] + t * 128 + ((unit[gi][e] ^ (uint32_t)(t & 7)) << 4));
            const uint16_t vb = *reinterpret_cast<const uint16_t*>(
                slab + base[gi][e + 1] + t * 128 + ((unit[gi][e + 1] ^ (uint32_t)(t & 7)) << 4));
            w[e / 2] = (uint32_t)va | ((uint32_t)vb << 16);
          }
          *reinterpret_cast<uint4*>(out + (size_t)(t0 + t) * d + g * 8) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      mbar_arrive(empty + buf);
    }
  }
}

}  // namespace

bool permute_supported(int d) {
  return d % 64 == 0 && d <= 8 * kPermWorkers * 4 && permute_rows(d) > 0;
}

poetx_status permute_cols_bf16(const void* in, void* out, const int32_t* perm, int T, int d,
                               cudaStream_t s) {
  if (T <= 0) return POETX_OK;
  if (!permute_supported(d)) return POETX_ERR_UNSUPPORTED;
  const int TM = permute_rows(d);
  CUtensorMap tin;
  if (!make_tmap_2d(&tin, in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d,
                    (uint32_t)TM, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return POETX_ERR_CUDA;
  const int sms = device_sm_count();
  const int n_slabs = (T + TM - 1) / TM;
  const int grid = n_slabs < sms ? n_slabs : sms;
  const int smem = 2 * TM * d * 2 + 1024 + 64;
  set_max_dynamic_smem((const void*)permute_kernel, smem);
  {
    KernelScope ks_("tc_permute_cols", s);
    permute_kernel<<<grid, kPermThreads, smem, s>>>(tin, static_cast<__nv_bfloat16*>(out), perm, T,
                                                    d, TM, device_error_word());
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
