// tc_blockapply.cu -- permuted block-diagonal apply on the tensor cores.
//
// [POET-X §2.B-§2.C] ("POET-X: Memory-efficient LLM Training by Scaling
// Orthogonal Transformation", gist.science summary, sections 2.B and 2.C):
// the orthogonal factors are block-diagonal, each block a small matrix of its
// own, and permutations are applied as index maps, never as matrices.  For
// every token t and block j this kernel computes
//     out_j[t][i] = sum_k Qop_j[i][k] * in_j[t][k],   Qop_j = Q_j or Q_j^T,
// in one of two forms:
//   GATHER_IN   in_j[t][k] = in[t][perm[j*b + k]],  out[t][j*b + i] = out_j[t][i]
//               (u = x_pi . B_P^T and g_z = dy_pi . B_R)
//   SCATTER_OUT in_j[t][k] = in[t][j*b + k],        out[t][perm[j*b + i]] = out_j[t][i]
//               (y = scatter(z . B_R^T) and dX = scatter(g_u . B_P))
// A permutation acts on the feature axis of token-major rows, so a CTA owns a
// slab of TM whole rows in shared memory (the gathered input slab, or the
// output slab being scattered into); no permuted copy of an activation ever
// exists in HBM.  The product runs as tcgen05.mma with M = 128 output
// features (Q from TMA, 128-byte swizzle), N = TM tokens, K = 16, fp32
// accumulators in TMEM.
//
// Roles (320 threads): warp 0 lane 0 issues TMA (slab or input tiles, and
// the Q chunks through an S-stage ring); warp 1 lane 0 issues the MMAs;
// warps 2..9 gather the per-block operand from the slab (GATHER_IN) and
// drain TMEM (both forms).  All waits are bounded.
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

constexpr int kThreads = 320;
constexpr int kWorkers = 256;          // warps 2..9
constexpr int kQChunk = 128 * 64 * 2;  // one A chunk: 128 output rows x 64 k, bf16
constexpr int kSmemMax = 232448;       // 227 KB opt-in maximum per CTA
constexpr int kMaxStages = 6;

struct Geo {
  int TM;          // tokens per slab (MMA N)
  int slab_bytes;  // TM x d bf16
  int bbuf_bytes;  // TM x b bf16 (one operand buffer)
  int stages;      // Q ring depth
  int smem;        // dynamic shared memory requested
};

Geo geometry(int d, int b) {
  Geo g;
  g.TM = (d <= 2048) ? 32 : 16;
  g.slab_bytes = g.TM * d * 2;
  g.bbuf_bytes = g.TM * b * 2;
  const int fixed = g.slab_bytes + 2 * g.bbuf_bytes + 1024 + 512;
  g.stages = (kSmemMax - fixed) / kQChunk;
  if (g.stages > kMaxStages) g.stages = kMaxStages;
  g.smem = fixed + g.stages * kQChunk;
  return g;
}

// bulk copy shared -> global (async proxy), one bulk group per call
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void worker_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory");
}

template <int TM>
__device__ __forceinline__ void tmem_ld_tokens(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  if constexpr (TM == 32) {
    tmem_ld32(taddr, r);
  } else {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
  }
  tmem_ld_wait();
#pragma unroll
  for (int t = 0; t < TM; ++t) v[t] = __uint_as_float(r[t]);
}

// Byte offset of element (row r, feature k) in a K-major operand laid out as
// 64-feature atom columns of [rows x 128 B] with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_offset(int r, int k, int rows) {
  return (uint32_t)((k >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

template <int TM, bool GATHER_IN>
__global__ void __launch_bounds__(kThreads, 1)
    blockapply_kernel(const __grid_constant__ CUtensorMap tmIn,
                      const __grid_constant__ CUtensorMap tmQ, __nv_bfloat16* __restrict__ out,
                      const int32_t* __restrict__ perm, int T, int d, int b, int transpose_q,
                      int stages, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int slab_bytes = TM * d * 2;
  const int bbuf_bytes = TM * b * 2;
  uint8_t* slab = smem;                       // GATHER_IN: input slab; SCATTER_OUT: output slab
  uint8_t* bbuf = smem + slab_bytes;          // 2 operand buffers
  uint8_t* qring = bbuf + 2 * bbuf_bytes;     // Q chunk ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(qring + stages * kQChunk);
  uint64_t* qfull = bars;
  uint64_t* qempty = qfull + kMaxStages;
  uint64_t* bfull = qempty + kMaxStages;
  uint64_t* bempty = bfull + 2;
  uint64_t* dfull = bempty + 2;
  uint64_t* dempty = dfull + 2;
  uint64_t* slab_full = dempty + 2;
  uint64_t* slab_empty = slab_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(slab_empty + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nb = d / b;
  const int halves = b / 128;
  const int kchunks = b / 64;
  const int n_slabs = (T + TM - 1) / TM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(qfull + s, 1);
      mbar_init(qempty + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bfull + i, GATHER_IN ? kWorkers : 1);
      mbar_init(bempty + i, 1);
      mbar_init(dfull + i, 1);
      mbar_init(dempty + i, kWorkers);
    }
    mbar_init(slab_full, 1);
    mbar_init(slab_empty, kWorkers);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int st = 0;
      uint32_t qph = 0;
      int jg = 0;
      bool ok = true;
      for (int it = 0, s = blockIdx.x; s < n_slabs && ok; s += gridDim.x, ++it) {
        const int t0 = s * TM;
        if (GATHER_IN) {
          if (!(ok = mbar_wait(slab_empty, (it & 1) ^ 1, err))) break;
          mbar_arrive_expect_tx(slab_full, slab_bytes);
          for (int c = 0; c < d / 64; ++c)
            tma_load_2d(slab + c * TM * 128, &tmIn, c * 64, t0, slab_full);
        }
        for (int j = 0; j < nb && ok; ++j, ++jg) {
          if (!GATHER_IN) {
            const int buf = jg & 1;
            if (!(ok = mbar_wait(bempty + buf, ((jg >> 1) & 1) ^ 1, err))) break;
            mbar_arrive_expect_tx(bfull + buf, bbuf_bytes);
            for (int c = 0; c < kchunks; ++c)
              tma_load_2d(bbuf + buf * bbuf_bytes + c * TM * 128, &tmIn, j * b + c * 64, t0,
                          bfull + buf);
          }
          for (int h = 0; h < halves && ok; ++h)
            for (int kc = 0; kc < kchunks; ++kc) {
              if (!(ok = mbar_wait(qempty + st, qph ^ 1, err))) break;
              mbar_arrive_expect_tx(qfull + st, kQChunk);
              uint8_t* dst = qring + st * kQChunk;
              if (!transpose_q) {
                // A[i][k] = Q[i][k]: 128 rows (i) x 64 k, K-major
                tma_load_2d(dst, &tmQ, kc * 64, j * b + h * 128, qfull + st);
              } else {
                // A[i][k] = Q[k][i]: 64 rows (k) x 64 i, twice, MN-major
                tma_load_2d(dst, &tmQ, h * 128, j * b + kc * 64, qfull + st);
                tma_load_2d(dst + 8192, &tmQ, h * 128 + 64, j * b + kc * 64, qfull + st);
              }
              if (++st == stages) { st = 0; qph ^= 1; }
            }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, TM, transpose_q != 0, false);
      int st = 0;
      uint32_t qph = 0;
      int jg = 0;
      bool ok = true;
      for (int s = blockIdx.x; s < n_slabs && ok; s += gridDim.x) {
        for (int j = 0; j < nb && ok; ++j, ++jg) {
          const int buf = jg & 1;
          const uint32_t par = (jg >> 1) & 1;
          if (!(ok = mbar_wait(bfull + buf, par, err))) break;
          if (!(ok = mbar_wait(dempty + buf, par ^ 1, err))) break;
          tc_fence_after();
          const uint32_t b_base = smem_u32(bbuf + buf * bbuf_bytes);
          for (int h = 0; h < halves && ok; ++h) {
            const uint32_t d_tmem = tmem_base + (uint32_t)((buf * 2 + h) * TM);
            for (int kc = 0; kc < kchunks; ++kc) {
              if (!(ok = mbar_wait(qfull + st, qph, err))) break;
              tc_fence_after();
              const uint32_t a_base = smem_u32(qring + st * kQChunk);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t adesc = transpose_q ? sw128_desc(a_base + kk * 2048, 8192, 1024)
                                                   : sw128_desc(a_base + kk * 32, 16, 1024);
                const uint64_t bdesc =
                    sw128_desc(b_base + kc * TM * 128 + kk * 32, 16, 1024);
                mma_bf16(d_tmem, adesc, bdesc, idesc, (kc | kk) != 0);
              }
              mma_commit(qempty + st);
              if (++st == stages) { st = 0; qph ^= 1; }
            }
          }
          mma_commit(bempty + buf);
          mma_commit(dfull + buf);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ workers
    const int wt = threadIdx.x - 64;          // 0..255
    const int quarter = warp % 4;
    const int h_mine = (warp - 2) / 4;        // output half drained by this warp
    int jg = 0;
    bool ok = true;
    bool pending_store = false;
    int prev_t0 = 0, prev_j = 0;
    auto drain = [&](int jdone, int j_of, int t0_of) {
      // epilogue of global block index jdone (block j_of of the slab at t0_of)
      const int buf = jdone & 1;
      if (!(ok = ok && mbar_wait(dfull + buf, (jdone >> 1) & 1, err))) return;
      tc_fence_after();
      if (h_mine < halves) {
        float v[32];
        tmem_ld_tokens<TM>(tmem_base + (uint32_t)((buf * 2 + h_mine) * TM) +
                               ((uint32_t)(quarter * 32) << 16),
                           v);
        const int i = h_mine * 128 + quarter * 32 + lane;
        if (GATHER_IN) {
          __nv_bfloat16* o = out + (size_t)t0_of * d + (size_t)j_of * b + i;
#pragma unroll
          for (int t = 0; t < TM; ++t)
            if (t0_of + t < T) o[(size_t)t * d] = __float2bfloat16_rn(v[t]);
        } else {
          __nv_bfloat16* os = reinterpret_cast<__nv_bfloat16*>(slab) + __ldg(perm + j_of * b + i);
#pragma unroll
          for (int t = 0; t < TM; ++t) os[(size_t)t * d] = __float2bfloat16_rn(v[t]);
        }
      }
      tc_fence_before();
      mbar_arrive(dempty + buf);
    };
    if (GATHER_IN) {
      // gather block j while the MMA works on block j-1, then drain block j-1
      for (int it = 0, s = blockIdx.x; s < n_slabs && ok; s += gridDim.x, ++it) {
        const int t0 = s * TM;
        if (!(ok = mbar_wait(slab_full, it & 1, err))) break;
        for (int j = 0; j < nb && ok; ++j, ++jg) {
          const int buf = jg & 1;
          if (!(ok = mbar_wait(bempty + buf, ((jg >> 1) & 1) ^ 1, err))) break;
          // unit (t, k8) = 8 consecutive k of token t, written as one 16-byte store;
          // lanes take 8 tokens x 4 k-groups, so the 8 tokens reading one
          // column of the swizzled slab hit 8 different banks
          uint8_t* dst = bbuf + buf * bbuf_bytes;
          const int units = TM * (b / 8);
          for (int u = wt; u < units; u += kWorkers) {
            const int tl = u & 7, kq = (u >> 3) & 3, rest = u >> 5;
            const int t = (rest % (TM / 8)) * 8 + tl;
            const int k8 = (rest / (TM / 8)) * 4 + kq;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const int c0 = __ldg(perm + j * b + k8 * 8 + e);
              const int c1 = __ldg(perm + j * b + k8 * 8 + e + 1);
              const uint16_t v0 = *reinterpret_cast<const uint16_t*>(
                  slab + (c0 >> 6) * TM * 128 + t * 128 + ((((c0 & 63) >> 3) ^ (t & 7)) << 4) +
                  (c0 & 7) * 2);
              const uint16_t v1 = *reinterpret_cast<const uint16_t*>(
                  slab + (c1 >> 6) * TM * 128 + t * 128 + ((((c1 & 63) >> 3) ^ (t & 7)) << 4) +
                  (c1 & 7) * 2);
              w[e / 2] = (uint32_t)v0 | ((uint32_t)v1 << 16);
            }
            *reinterpret_cast<uint4*>(dst + sw128_offset(t, k8 * 8, TM)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          mbar_arrive(bfull + buf);
          if (j == nb - 1) mbar_arrive(slab_empty);   // the slab is no longer read
          if (jg > 0) drain(jg - 1, prev_j, prev_t0);
          prev_j = j;
          prev_t0 = t0;
        }
      }
      if (ok && jg > 0) drain(jg - 1, prev_j, prev_t0);
    } else {
      // drain each block into the output slab, then store the slab's rows
      for (int s = blockIdx.x; s < n_slabs && ok; s += gridDim.x) {
        const int t0 = s * TM;
        if (pending_store) {
          // the previous slab's bulk store must have finished reading it
          if (wt == 0) bulk_wait_read();
          worker_bar();
          pending_store = false;
        }
        for (int j = 0; j < nb && ok; ++j, ++jg) drain(jg, j, t0);
        if (!ok) break;
        fence_proxy_async_smem();
        worker_bar();
        if (wt == 0) {
          const int rows = min(TM, T - t0);
          bulk_store(out + (size_t)t0 * d, slab, (uint32_t)(rows * d * 2));
        }
        pending_store = true;
      }
      if (wt == 0 && pending_store) bulk_wait_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 128);
  }
}

}  // namespace

bool blockapply_supported(int d, int b) {
  if (b != 128 && b != 256) return false;
  if (d % b != 0 || d % 64 != 0) return false;
  const Geo g = geometry(d, b);
  return g.stages >= 2;
}

// GATHER_IN  (scatter == false): out[t][jb+i] = sum_k Qop_j[i][k] in[t][perm[jb+k]]
// SCATTER_OUT(scatter == true):  out[t][perm[jb+i]] = sum_k Qop_j[i][k] in[t][jb+k]
poetx_status blockapply_bf16(const void* in, void* out, const void* Q, const int32_t* perm, int T,
                             int d, int b, bool transpose_q, bool scatter, cudaStream_t s) {
  if (T <= 0) return POETX_OK;
  if (!blockapply_supported(d, b)) return POETX_ERR_UNSUPPORTED;
  const Geo g = geometry(d, b);
  CUtensorMap tin, tq;
  if (!make_tmap_2d(&tin, in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d,
                    (uint32_t)g.TM, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return POETX_ERR_CUDA;
  const int nb = d / b;
  const bool okq =
      transpose_q ? make_tmap_2d(&tq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)nb * b,
                                 (uint64_t)b, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)
                  : make_tmap_2d(&tq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)nb * b,
                                 (uint64_t)b, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!okq) return POETX_ERR_CUDA;
  const int sms = device_sm_count();
  const int n_slabs = (T + g.TM - 1) / g.TM;
  const int grid = n_slabs < sms ? n_slabs : sms;
  int* err = device_error_word();
  const char* name = scatter ? "tc_blockapply_scatter" : "tc_blockapply_gather";
  auto launch = [&](auto kern) {
    set_max_dynamic_smem((const void*)kern, g.smem);
    KernelScope ks_(name, s);
    kern<<<grid, kThreads, g.smem, s>>>(tin, tq, (__nv_bfloat16*)out, perm, T, d, b,
                                        transpose_q ? 1 : 0, g.stages, err);
  };
  if (g.TM == 32) {
    if (scatter) launch(blockapply_kernel<32, false>);
    else launch(blockapply_kernel<32, true>);
  } else {
    if (scatter) launch(blockapply_kernel<16, false>);
    else launch(blockapply_kernel<16, true>);
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
