// tc_exchange.cuh -- the cluster-wide feature exchange behind every permuted operand.
//
// [POET-X §2.B] ("POET-X: Memory-efficient LLM Training by Scaling
// Orthogonal Transformation", gist.science summary, section 2.B): the
// permutations are index maps, applied while data moves, never as a permuted
// copy of an activation in HBM.  A cluster of C CTAs works on one tile of TT
// tokens at a time; CTA c owns the natural feature columns [c*F, (c+1)*F) of
// the permuted tensor and the blocks [c*G, (c+1)*G).  A permuted feature row
// (the TT tokens of one feature, 128 bytes) travels once: the CTA that loaded
// it writes it straight to its place in a small per-cluster exchange ring in
// the workspace (a few MB, rewritten every few microseconds, so it stays in
// L2), and the CTA that needs it fetches its whole part of the slot with one
// bulk copy.  Hand-offs are cluster mbarriers (waited on by polling):
//   x_full[slot] of the reader: C remote arrivals, one per writer CTA,
//                               released by its loader warp once the CTA's
//                               writers have stored their rows (a local
//                               barrier, so the writers never wait on the
//                               release);
//   x_free[slot] of the writer: C remote arrivals, one per reader, after the
//                               reader's bulk copy of its part has landed --
//                               sent only for slots that will be written
//                               again, so every remote arrive is waited for by
//                               its target and none is in flight at the end.
// Every wait is bounded (tc_ptx.cuh).
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace poetx {
namespace tc {
namespace xchg {

constexpr int TT = 64;          // tokens per tile (the epilogues hold a tile row in two 32-wide TMEM loads)
constexpr int kMovers = 256;    // threads that write feature rows (warps 2..9)
constexpr int kMaxSlots = 4;    // exchange slots in the workspace ring (at most; 4 measured
                                // faster than 8 or 6 at the square 2048 layer: less L2 held)
constexpr int kTableOff = 512;  // routing table, after the barrier block

__device__ __forceinline__ void movers_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kMovers) : "memory");
}

__device__ __forceinline__ uint4 pack8f(const float* v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// Barrier block at the start of shared memory (uint64 words; under kTableOff bytes).
struct Bars {
  uint64_t* s_full;     // [4] own-column input tile landed (TMA)
  uint64_t* s_empty;    // [4] own-column input tile consumed
  uint64_t* x_full;     // [8] every writer has written this CTA's part of an exchange slot
  uint64_t* x_free;     // [8] every reader has fetched its part of an exchange slot
  uint64_t* r_full;     // [4] fetched part landed in shared memory
  uint64_t* r_empty;    // [4] fetched part consumed
  uint64_t* a_full;     // [2] accumulators ready
  uint64_t* a_empty;    // [2] accumulators drained
  uint64_t* q_full;     // [1] one-time operand staged (Q blocks; the dQ sums)
  uint64_t* v_full;     // [4] second, unpermuted operand landed (TMA)
  uint64_t* v_empty;    // [4] second operand consumed
  uint64_t* moved;      // [8] this CTA's writers have stored their rows of an exchange slot
  uint64_t* q_done;     // [1] the one-time operand is in tensor memory (128 arrivals)
  uint32_t* tmem_slot;
};

__device__ __forceinline__ Bars bars_at(uint8_t* smem) {
  uint64_t* b = reinterpret_cast<uint64_t*>(smem);
  Bars r;
  r.s_full = b;
  r.s_empty = b + 4;
  r.x_full = b + 8;
  r.x_free = b + 16;
  r.r_full = b + 24;
  r.r_empty = b + 28;
  r.a_full = b + 32;
  r.a_empty = b + 34;
  r.q_full = b + 36;
  r.v_full = b + 37;
  r.v_empty = b + 41;
  r.moved = b + 45;
  r.q_done = b + 53;
  r.tmem_slot = reinterpret_cast<uint32_t*>(b + 54);   // 440 bytes in all, under kTableOff
  return r;
}

// s_empty arrivals: the movers (GATHER side) or an MMA commit (SCATTER side);
// r_empty: an MMA commit or one mover; moved: every thread that writes rows.
__device__ __forceinline__ void init_bars(const Bars& br, int C, uint32_t s_empty_count,
                                          uint32_t r_empty_count, uint32_t writers) {
  for (int i = 0; i < kMaxSlots; ++i) {
    mbar_init(br.x_full + i, (uint32_t)C);
    mbar_init(br.x_free + i, (uint32_t)C);
    mbar_init(br.moved + i, writers);
  }
  for (int i = 0; i < 4; ++i) {
    mbar_init(br.s_full + i, 1);
    mbar_init(br.s_empty + i, s_empty_count);
  }
  for (int i = 0; i < 4; ++i) {
    mbar_init(br.r_full + i, 1);
    mbar_init(br.r_empty + i, r_empty_count);
    mbar_init(br.v_full + i, 1);
    mbar_init(br.v_empty + i, 1);
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(br.a_full + i, 1);
    mbar_init(br.a_empty + i, 128);
  }
  mbar_init(br.q_full, 1);
  mbar_init(br.q_done, 128);
  fence_mbar_init();
}

// Remote arrive on barrier `bar` of CTA `who` of the cluster (0 <= who < C;
// callers with who >= C do nothing), so C threads signal the C CTAs in
// parallel.  With `release` the memory accesses the caller has made or
// observed (e.g. through a CTA barrier) are ordered before the arrival at
// cluster scope; without it the arrival is a pure signal.
__device__ __forceinline__ void arrive_one(uint64_t* bar, int who, int C, bool release) {
  if (who < C) {
    const uint32_t ra = mapa_shared(smem_u32(bar), (uint32_t)who);
    if (release) mbar_arrive_remote(ra);
    else mbar_arrive_remote_relaxed(ra);
  }
}

// Iterations (tiles) of cluster `cluster_id` when clusters take tiles round-robin.
__device__ __forceinline__ int cluster_iters(int cluster_id, int n_clusters, int n_tiles) {
  return cluster_id < n_tiles ? (n_tiles - cluster_id + n_clusters - 1) / n_clusters : 0;
}

// The loader (one thread): fetches this CTA's part of every exchange slot
// once all C writers have signalled it.  With `gate`, the first fetch also
// waits for that barrier's first phase (the fetch buffers held another
// operand until then).
__device__ __forceinline__ void loader_loop(const Bars& br, int NR, int NX, int r_bytes, uint8_t* rbuf,
                                            const uint8_t* part0, size_t slot_stride, int n_it,
                                            bool& ok, int* err, uint64_t* gate = nullptr) {
  if (gate && n_it > 0) ok = mbar_wait(gate, 0, err);
  for (int it = 0; it < n_it && ok; ++it) {
    const int r = it % NR, x = it % NX;
    if (!(ok = mbar_wait(br.r_empty + r, ((it / NR) & 1) ^ 1, err))) break;   // buffer free
    if (!(ok = mbar_wait_cluster(br.x_full + x, (it / NX) & 1, err))) break;  // slot written
    fence_proxy_async_global();
    mbar_arrive_expect_tx(br.r_full + r, (uint32_t)r_bytes);
    bulk_load_g2s(rbuf + r * r_bytes, part0 + (size_t)x * slot_stride, (uint32_t)r_bytes,
                  br.r_full + r);
  }
}

// The signalling warp (all 32 lanes call this): for every iteration, lanes
// 0..C-1 wait until this CTA's writers have stored their rows of the slot
// (local barrier `moved`) and then signal the C readers with a remote arrive
// on x_full, released at cluster scope (which carries the writers' stores the
// lane has observed).  The writers never wait for the release themselves.
__device__ __forceinline__ void signal_loop(const Bars& br, int NX, int n_it, int C, int lane,
                                            bool& ok, int* err) {
  for (int it = 0; it < n_it && ok; ++it) {
    const int x = it % NX;
    bool lok = true;
    if (lane < C && (lok = mbar_wait(br.moved + x, (it / NX) & 1, err)))
      arrive_one(br.x_full + x, lane, C, true);
    ok = __all_sync(0xffffffffu, lok);   // the lanes leave together
  }
}

// Reader side of a fetched slot: lanes 1..C of the calling warp tell the C
// writers that this CTA's part of iteration it's slot has been fetched, if a
// later iteration will write the slot again.
__device__ __forceinline__ void ack_fetch(const Bars& br, int it, int NX, int n_it, int who, int C) {
  if (it + NX < n_it) arrive_one(br.x_free + it % NX, who, C, false);
}

// Exchange slots per cluster ring, and the ring's size, for `clusters`
// clusters of C CTAs over n_tiles tiles: no more slots than iterations.
inline int ring_slots(int n_tiles, int clusters) {
  const int n_it = (n_tiles + clusters - 1) / clusters;
  return n_it < kMaxSlots ? (n_it > 0 ? n_it : 1) : kMaxSlots;
}

// Routing table of the GATHER side, one entry per owned natural feature f of
// CTA c: (reader CTA << 24) | byte offset of the feature's row in the
// reader's part, where the row sits at the feature's gathered position
// (block j = p / B, position k = p % B of p = inv[c*F + f]).
template <int B>
__device__ __forceinline__ void gather_table(uint32_t* table, const int32_t* __restrict__ inv, int c,
                                             int F, int G) {
  for (int f = threadIdx.x; f < F; f += blockDim.x) {
    const int p = __ldg(inv + c * F + f);
    const int j = p / B, k = p % B;
    table[f] = ((uint32_t)(j / G) << 24) | (uint32_t)(((j % G) * B + k) * 128);
  }
}

// One mover thread (pt = 0..kMovers-1) on one input tile S (the CTA's F
// natural columns of TT tokens, F/64 TMA boxes of [TT tokens][64 features],
// 128-byte swizzle): for each of its features collects the TT tokens (placed
// in the row's 128-byte swizzle order) and writes the row into the part of
// the CTA owning the feature's block.
__device__ __forceinline__ void move_gather_rows(const uint8_t* S, uint8_t* slot, const uint32_t* table,
                                                 int F, int r_bytes, int pt) {
  for (int f = pt; f < F; f += kMovers) {
    const uint32_t ent = table[f];
    const uint32_t roff = ent & 0xFFFFFFu;
    const uint32_t k7 = (roff >> 7) & 7u;
    uint8_t* row = slot + (size_t)(ent >> 24) * r_bytes + roff;
#pragma unroll
    for (int grp = 0; grp < TT / 8; ++grp) {
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int tr = grp * 8 + e;
        const uint32_t off = (uint32_t)((f >> 6) * (TT * 128) + tr * 128 +
                                        ((((f >> 3) & 7) ^ (tr & 7)) << 4) + (f & 7) * 2);
        v[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(S + off));
      }
      *reinterpret_cast<uint4*>(row + ((((uint32_t)grp) ^ k7) << 4)) = pack8f(v);
    }
  }
}

}  // namespace xchg
}  // namespace tc
}  // namespace poetx
