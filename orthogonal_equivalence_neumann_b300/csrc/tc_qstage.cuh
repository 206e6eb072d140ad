// tc_qstage.cuh -- a CTA's Q blocks into tensor memory, as the A operand of its block products.
//
// The block-diagonal factors of "POET-X: Memory-efficient LLM Training by
// Scaling Orthogonal Transformation" (gist.science summary, section 2.C) are
// applied block by block; a kernel that applies the same few blocks to many
// token tiles keeps their Qop (Q or Q^T) resident in tensor memory for the
// whole launch, so tcgen05.mma reads A from TMEM and only the activations
// stream.  Staging: one thread brings the blocks into shared memory by TMA
// (128-byte swizzled 64 x 64 boxes, which make both the row reads and the
// column reads below conflict-free); four warps (one per TMEM lane quarter)
// then write Qop_j into tensor memory: lanes = output rows i, two bf16 of
// consecutive k per 32-bit column, block jj's half h at column
// (jj * B/128 + h) * B/2.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace poetx {
namespace tc {

// Issues the TMA loads of blocks [j0, j0 + G) of Q into `stage` (G * B * B * 2
// bytes), completing on q_full.
__device__ __forceinline__ void issue_q_loads(const CUtensorMap* tmQ, uint8_t* stage, int j0, int G,
                                              int B, uint64_t* q_full) {
  mbar_arrive_expect_tx(q_full, (uint32_t)(G * B * B * 2));
  for (int jj = 0; jj < G; ++jj)
    for (int rb = 0; rb < B / 64; ++rb)
      for (int cb = 0; cb < B / 64; ++cb)
        tma_load_2d(stage + jj * (B * B * 2) + cb * (B * 128) + rb * (64 * 128), tmQ, cb * 64,
                    (j0 + jj) * B + rb * 64, q_full);
}

// Byte offset of Q[row][col] in the staged block.
template <int B>
__device__ __forceinline__ uint32_t qst_off(int row, int col) {
  return (uint32_t)((col >> 6) * (B * 128) + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                    (col & 7) * 2);
}

template <int B>
__device__ void q_stage_to_tmem(const uint8_t* stage, int G, int transpose_q, uint32_t tmem_base,
                                int quarter, int lane) {
  constexpr int halves = B / 128;
  for (int jj = 0; jj < G; ++jj)
    for (int h = 0; h < halves; ++h) {
      const int i = h * 128 + quarter * 32 + lane;
      const uint8_t* blk = stage + (size_t)jj * B * B * 2;
      const uint32_t col0 = (uint32_t)((jj * halves + h) * (B / 2));
      for (int c = 0; c < B / 2; c += 32) {
        uint32_t r[32];
        if (transpose_q) {
          // row i of Q^T is column i of Q: lanes read consecutive columns of one row
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k = 2 * (c + e);
            const uint16_t lo = *reinterpret_cast<const uint16_t*>(blk + qst_off<B>(k, i));
            const uint16_t hi = *reinterpret_cast<const uint16_t*>(blk + qst_off<B>(k + 1, i));
            r[e] = (uint32_t)lo | ((uint32_t)hi << 16);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 v = *reinterpret_cast<const uint4*>(blk + qst_off<B>(i, 2 * c + 8 * q));
            r[4 * q] = v.x; r[4 * q + 1] = v.y; r[4 * q + 2] = v.z; r[4 * q + 3] = v.w;
          }
        }
        tmem_st32(tmem_base + col0 + (uint32_t)c + ((uint32_t)(quarter * 32) << 16), r);
      }
    }
  tmem_st_wait();
}

}  // namespace tc
}  // namespace poetx
