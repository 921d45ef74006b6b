// Tensor-core attention forward for sm_103a: the tiled, fused method of "I/O-Aware Kernels"
// (datasystem.school, Module 5), section "FlashAttention: tiling + online softmax". A query tile
// stays in shared memory, key/value tiles stream through a TMA-fed ring, S = Q K^T and O += P V run
// as tcgen05 MMAs with their accumulators in tensor memory (TMEM), and the softmax is computed
// online (running max m, running sum l, rescaled O), so no score ever reaches device memory.
//
// One kernel serves the dense layout and the paged/ragged layout of the page's section
// "FlashInfer: I/O-aware attention for serving"; they differ only in how tiles are addressed.
// On the paged layout it also packs the query heads of a GQA group into one tile (rows = token x
// head) and can split each unit's keys into ranges written as fp32 partial states, which makes it
// the path for prefill, chunked prefill, multi-token verify and decode alike.
//
// The grid has one CTA per work item, and a CTA that finishes its item takes over the item of a
// CTA that has not started yet (cluster launch control), so an SM pays the CTA set-up once while
// items still run in the launch order the units are numbered in.
//
// CTA organisation (384 threads, one CTA per SM):
//   warp 0      TMA producer: Q tiles once, then K_0, V_0, K_1, V_1, ... into a ring of stages
//   warp 1      TMEM owner; one lane issues every tcgen05.mma of query tile 0
//   warp 2      one lane issues every tcgen05.mma of query tile 1
//   warp 3      paged layout: second TMA producer (the V tiles; warp 0 then loads Q and K); dense: idle
//   warps 4-7   softmax warpgroup 0 -> query tile 0 (rows 0..127 of the CTA's 256)
//   warps 8-11  softmax warpgroup 1 -> query tile 1 (rows 128..255)
// The two warpgroups ping-pong: while one computes its softmax the tensor core runs the other's
// P V and next Q K^T (the two MMA issuers take turns to keep that order).
//
// TMEM columns: S/P of tile g at [128 g, 128 g + 128) (P, as packed bf16 pairs, overwrites the
// first 64 columns of S), O of tile g at [256 + g D, 256 + (g+1) D). At d = 64, P of tile g has
// columns [384 + 64 g, 448 + 64 g) of its own: the issuer then puts a tile's next Q K^T ahead of
// its P V as soon as the softmax has read S, and the issuers do not take turns.
#include <cuda_bf16.h>
#include <atomic>
#include <cstdlib>
#include "kernels.cuh"

namespace fa {

namespace {

// A rescale of O is deferred until the running maximum grows by more than 2^8: until then the
// stale maximum is kept, so P entries stay below 256 (exact in fp32 and well inside bf16 range).
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kBM * D * 2;  // one 128-row tile of Q, K or V (bf16)
  static constexpr int kSub = D / 64;             // 128-byte-wide column blocks per tile
  static constexpr int kSubBytes = kBM * 128;     // 16 KB per column block
  static constexpr int kStages = D == 128 ? 5 : 8;
  static constexpr int kSmemBytes = 1024 + (kQTiles + kStages) * kTileBytes;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
};

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

// Wait sites recorded in the device status word when a wait times out.
enum : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaQ = 2,
  kSiteMmaFull = 3,
  kSiteMmaP = 4,
  kSiteSoftmaxS = 5,
  kSiteSoftmaxO = 6,
  kSiteDrain = 7,
  kSiteMmaTurn = 8,
  kSiteTakeOver = 9,
  kSiteMmaSFree = 10,
  kSiteSoftmaxPV = 11,
};

// One unit of work: a pair of 128-row query tiles of one (sequence, query head), or, with GQA
// packing (paged, pack > 1), of one (sequence, kv head): tile row r is then query token r / pack
// of the tile and query head h + r % pack, so the pack heads sharing a kv head read each K/V tile
// once, and a sequence with few query tokens (verify, decode rows) still fills the tile.
struct Unit {
  int seq, h, hk, q_len, kv_len, off, nmax;
  int split, kv_t0;   // paged key split: this unit's split and its first key tile
  int64_t tok0;  // token index of the sequence's first query row
  int nkv[kQTiles];   // key tiles per query tile; -1 = the tile has no query rows
  int row0[kQTiles];  // first (packed) row of each tile within its sequence
};

template <bool PAGED>
__device__ __forceinline__ int count_units(const PrefillParams& p) {
  if constexpr (PAGED) {
    return *p.work_count * (p.Hq / p.pack) * p.kv_splits;
  } else {
    return ((p.S + 2 * kBM - 1) / (2 * kBM)) * p.B * p.Hq;
  }
}

// Unit u in the global order (paged: the order of the device-built work list; dense: below).
template <bool PAGED>
__device__ __forceinline__ void unit_at(const PrefillParams& p, int u, Unit& w) {
  int qt2;
  if constexpr (PAGED) {
    const int slots = p.Hq / p.pack;
    w.split = u % p.kv_splits;  // the splits of one tile pair are adjacent in the order
    const int rest = u / p.kv_splits;
    const int item = rest / slots;
    w.h = (rest % slots) * p.pack;  // the first query head of the tile
    const int2 it = p.work_list[item];
    w.seq = it.x;
    qt2 = it.y;
    const int c0 = p.cu_seqlens_q[w.seq], c1 = p.cu_seqlens_q[w.seq + 1];
    w.tok0 = c0;
    w.q_len = c1 - c0;
    w.kv_len = min(p.kv_lens[w.seq], p.max_pages_per_seq * p.page_size);
  } else {
    // Units are grouped by chunks of kv heads sized so that one chunk is about one wave of CTAs:
    // CTAs running together then read the K/V of only a few heads, which stay in L2 while every
    // query tile of those heads streams them. Inside a chunk: query tiles heaviest first (causal),
    // and for each tile the query heads of the chunk, those sharing a kv head adjacent.
    const int T = (p.S + 2 * kBM - 1) / (2 * kBM);
    const int G = p.group;
    const int NKV = p.B * p.Hkv;
    const int per_chunk = p.kv_heads_per_chunk * G * T;
    const int chunk = u / per_chunk;
    const int kv0 = chunk * p.kv_heads_per_chunk;
    const int width = min(p.kv_heads_per_chunk, NKV - kv0) * G;  // query heads in this chunk
    const int r = u - chunk * per_chunk;
    qt2 = p.causal ? (T - 1 - r / width) : (r / width);
    const int idx = r % width;
    const int kvh = kv0 + idx / G;
    w.seq = kvh / p.Hkv;
    w.h = (kvh % p.Hkv) * G + idx % G;
    w.tok0 = (int64_t)w.seq * p.S;
    w.q_len = p.S;
    w.kv_len = p.S;
    w.split = 0;
  }
  w.hk = w.h / p.group;
  w.off = w.kv_len - w.q_len;  // bottom-right causal alignment
  w.nmax = 0;
  const int pack = PAGED ? p.pack : 1;
#pragma unroll
  for (int g = 0; g < kQTiles; ++g) {
    w.row0[g] = qt2 * (2 * kBM) + g * kBM;
    if (w.row0[g] >= w.q_len * pack) {
      w.nkv[g] = -1;
    } else {
      const int last = min(w.row0[g] + kBM - 1, w.q_len * pack - 1) / pack;  // last query token
      const int lim = p.causal ? min(w.kv_len, last + w.off + 1) : w.kv_len;
      w.nkv[g] = lim > 0 ? (lim + kBN - 1) / kBN : 0;
    }
    w.nmax = max(w.nmax, w.nkv[g]);
  }
  w.kv_t0 = 0;
  if (PAGED && p.kv_splits > 1) {
    // split s takes key tiles [s * per, (s + 1) * per) of what each query tile needs
    const int per = ((w.kv_len + kBN - 1) / kBN + p.kv_splits - 1) / p.kv_splits;
    w.kv_t0 = w.split * per;
    w.nmax = 0;
#pragma unroll
    for (int g = 0; g < kQTiles; ++g) {
      if (w.nkv[g] >= 0) w.nkv[g] = max(0, min(w.nkv[g] - w.kv_t0, per));
      w.nmax = max(w.nmax, w.nkv[g]);
    }
  }
}

// S = Q K^T for one 128x128 tile: D/16 MMAs of K = 16. Shared-memory descriptors are built once
// by the caller; a K step only moves the start address, whose field (address >> 4, bits 0-13)
// never carries into the next field inside the CTA's shared memory, so each step adds a
// compile-time constant: 32 bytes inside a 128-byte swizzle row, and every 4 steps the next
// 16 KB column block.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (uint64_t)((kk >> 2) * (Cfg<D>::kSubBytes >> 4) + (kk & 3) * 2);
    mma_ss(d_tmem, a_desc + off, b_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V for one tile: P (bf16 pairs) from TMEM as A, V as the MN-major B operand; a K step
// of 16 keys is 16 rows of 128 bytes (2048 bytes) in each 64-column block of d, and P's 16 keys
// are 8 TMEM columns.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc, uint32_t idesc,
                                         uint32_t accumulate) {
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk)
    mma_ts(o_tmem, p_tmem + kk * 8, v_desc + (uint64_t)kk * (2048 >> 4), idesc, kk > 0 ? 1u : accumulate);
}

// Softmax numerators for 32-column chunks [C0, C0 + NC) of one score row held in registers:
// p = 2^(s * sl2 - m) with the affine step and the row sum on fp32 pairs, P packed to bf16 pairs
// and written to TMEM over the chunk's S columns (16 columns per chunk). Returns the chunks'
// partial row sum as two fp32 halves of a pair.
template <int C0, int NC>
__device__ __forceinline__ uint64_t softmax_chunks(const uint32_t* sr, float sl2, float neg_m, uint32_t tS) {
  const uint64_t sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(neg_m, neg_m);
  uint64_t ls4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int cc = C0; cc < C0 + NC; ++cc) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = cc * 32 + 2 * i;
      float x0, x1;
      split_f32x2(fma_f32x2(f32x2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2, negm2), x0, x1);
      const float p0 = ex2(x0), p1 = ex2(x1);
      ls4[i & 3] = add_f32x2(ls4[i & 3], f32x2(p0, p1));
      pk[i] = pack_bf16x2(p0, p1);
    }
    tmem_st16(tS + cc * 16, pk);
  }
  return add_f32x2(add_f32x2(ls4[0], ls4[1]), add_f32x2(ls4[2], ls4[3]));
}

// O rescale by alpha when a row's running maximum moved (rare: a loop that is not unrolled keeps
// the code small). Runs before the tile's P is released to the MMA: P V of the previous tile is
// complete, because the commit that signalled this tile's S was issued after it.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tO, bool any_need, float alpha) {
  if (!any_need) return;
  const uint64_t a2 = f32x2(alpha, alpha);
#pragma unroll 1
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t orr[32];
    tmem_ld32(tO + cc * 32, orr);
    tmem_ld_wait(orr);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float a, b;
      split_f32x2(mul_f32x2(f32x2(u2f(orr[2 * i]), u2f(orr[2 * i + 1])), a2), a, b);
      orr[2 * i] = f2u(a);
      orr[2 * i + 1] = f2u(b);
    }
    tmem_st32(tO + cc * 32, orr);
  }
}

// Softmax numerators of a whole 128-key score row held in registers, like softmax_chunks, with P
// left in registers (pk: bf16 pairs) for the caller to store. Returns the row sum as two halves.
__device__ __forceinline__ uint64_t softmax_regs(const uint32_t* sr, float sl2, float neg_m, uint32_t* pk) {
  const uint64_t sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(neg_m, neg_m);
  uint64_t ls4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int i = 0; i < kBN / 2; ++i) {
    float x0, x1;
    split_f32x2(fma_f32x2(f32x2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), sl2x2, negm2), x0, x1);
    const float p0 = ex2(x0), p1 = ex2(x1);
    ls4[i & 3] = add_f32x2(ls4[i & 3], f32x2(p0, p1));
    pk[i] = pack_bf16x2(p0, p1);
  }
  return add_f32x2(add_f32x2(ls4[0], ls4[1]), add_f32x2(ls4[2], ls4[3]));
}

// Row max of 32-column chunks [C0, C0 + NC): four independent chains of three-input max.
template <int C0, int NC>
__device__ __forceinline__ float row_max_chunks(const uint32_t* sr) {
  float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c = C0 * 32; c < (C0 + NC) * 32; c += 2)
    mx4[(c >> 1) & 3] = max3f(mx4[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
  return max3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
}

// Persistent schedule: CTA c takes units c, 2G-1-c, 2G+c, 4G-1-c, ... (a snake over the
// heaviest-first order, so every CTA gets a similar share of heavy and light units).
__device__ __forceinline__ int unit_of_round(int r) {
  const int G = gridDim.x, c = blockIdx.x;
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// Work items of the dense launches: one unit, or under causal masking a mirrored pair of units —
// query-tile pair i and its mirror T-1-i of one query head, heaviest first. Every pair then costs
// the same, so CTAs stay balanced. Sets u0 and u1 to the item's units as indices of the dense order
// (unit_at); -1 where the item has no such unit.
template <bool PAGED>
__device__ __forceinline__ void item_units(const PrefillParams& p, int item, int n_units, int& u0, int& u1) {
  u1 = -1;
  if (!p.pair_units) {
    u0 = item < n_units ? item : -1;
    return;
  }
  if constexpr (PAGED) {
    u0 = -1;
  } else {
    const int T = (p.S + 2 * kBM - 1) / (2 * kBM);
    const int half = (T + 1) / 2;  // pairs per query head
    const int G = p.group;
    const int NKV = p.B * p.Hkv;
    const int pairs_per_chunk = p.kv_heads_per_chunk * G * half;
    const int chunk = item / pairs_per_chunk;
    const int kv0 = chunk * p.kv_heads_per_chunk;
    const int width = min(p.kv_heads_per_chunk, NKV - kv0) * G;
    const int rc = item - chunk * pairs_per_chunk;
    const int i = rc / width, head = rc % width;
    const int chunk_start = chunk * p.kv_heads_per_chunk * G * T;
    u0 = chunk_start + i * width + head;                                       // qt2 = T-1-i
    if (T - 1 - i != i) u1 = chunk_start + (T - 1 - i) * width + head;          // qt2 = i
  }
}

// Launch cancellation state shared by the warps that walk the units: two response slots, each
// with a full barrier (the response's 16 bytes) and an empty barrier (one arrival per walker).
struct TakeOver {
  uint4 resp[2];
  uint64_t full[2], empty[2];
};
constexpr int kUnitWalkers = 11;  // warps 0-2 and 4-11 (and warp 3 on the paged layout)

// Which units a CTA runs, in the same sequence in every warp. A persistent launch walks the snake
// order of unit_of_round. Otherwise a CTA runs work item blockIdx.x; with TAKE, once its item is
// done it takes over the item of a CTA that has not started yet: the producer requests a launch
// cancellation while it loads the item's last unit, and every walker reads the response. CTAs then run items in the hardware's launch order (which keeps the
// L2-aware unit order) while a CTA's set-up — barriers, TMEM, the first loads — is paid once per
// SM rather than once per item, and the next item's first loads overlap this item's tail.
struct Cursor {
  int u0, u1;      // the current item's units (-1: none)
  int sub;         // units of the current item handed out so far
  uint32_t taken;  // responses read so far
  // true once the current item has no unit left to hand out
  __device__ __forceinline__ bool item_done() const { return sub >= 2 || (sub == 1 && u1 < 0); }
};

template <bool PAGED>
__device__ __forceinline__ Cursor first_cursor(const PrefillParams& p, int n_units) {
  Cursor c{-1, -1, 0, 0u};
  item_units<PAGED>(p, (int)blockIdx.x, n_units, c.u0, c.u1);
  return c;
}

template <bool PAGED, bool TAKE>
__device__ __forceinline__ int next_unit(const PrefillParams& p, Cursor& c, int r, int n_units, TakeOver& t,
                                         volatile int* abort) {
  if constexpr (!TAKE) {
    if (p.pair_units) return r == 0 ? c.u0 : (r == 1 ? c.u1 : -1);
    const int u = unit_of_round(r);
    return u < n_units ? u : -1;
  } else {
    if (!c.item_done()) return c.sub++ == 0 ? c.u0 : c.u1;
    const uint32_t s = c.taken & 1, parity = (c.taken >> 1) & 1;
    ++c.taken;
    int item = -1;
    if (mbar_wait(&t.full[s], parity, abort, p.status, kSiteTakeOver)) item = launch_cancel_result(&t.resp[s]);
    item = __shfl_sync(0xffffffffu, item, 0);  // lane 0 decides for its warp
    if ((threadIdx.x & 31) == 0) mbar_arrive(&t.empty[s]);
    // A failed request, or an item without units (a grid that is an upper bound ends with such
    // items), ends the walk: the producer asks for another item only after loading a unit.
    c.u0 = -1;
    if (item >= 0) item_units<PAGED>(p, item, n_units, c.u0, c.u1);
    c.sub = 1;
    return c.u0;
  }
}

template <int D, bool PAGED, bool TAKE>
__global__ void __launch_bounds__(kPrefillThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = Cfg<D>;
  constexpr int NS = C::kStages;
  constexpr int TB = C::kTileBytes;
  // d = 64 leaves 128 TMEM columns free (S 2 x 128 and O 2 x 64 of 512): P gets a region of its
  // own there instead of overwriting S, so each tile's next Q K^T is issued as soon as the softmax
  // has read S, ahead of this tile's P V (the next scores are ready when the softmax is)
  constexpr bool kSepP = D == 64;
  constexpr uint32_t kColP = 384;  // kSepP: P of query tile g at columns 384 + 64 g (bf16 pairs)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                  // kQTiles tiles
  uint8_t* sKV = smem + kQTiles * TB;  // NS stages

  __shared__ uint64_t bar_q_full, bar_q_empty, bar_full[NS], bar_empty[NS];
  __shared__ uint64_t bar_s[kQTiles], bar_p[kQTiles], bar_o[kQTiles], bar_o_free[kQTiles], bar_drain[kQTiles];
  __shared__ uint64_t bar_sfree[kQTiles], bar_pv[kQTiles];  // separate P (d = 64) only
  __shared__ uint64_t bar_turn[2];
  __shared__ alignas(16) TakeOver take;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_units = count_units<PAGED>(p);
  if (!p.pair_units && (int)blockIdx.x >= n_units) return;  // the grid is an upper bound

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, kQTiles);  // one arrival per MMA issuer
#pragma unroll
    for (int g = 0; g < kQTiles; ++g) {
      mbar_init(&bar_s[g], 1);
      mbar_init(&bar_sfree[g], 4 * 32);
      mbar_init(&bar_pv[g], 1);
      mbar_init(&bar_p[g], 4 * 32);
      mbar_init(&bar_o[g], 1);
      mbar_init(&bar_o_free[g], 4 * 32);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], kQTiles);  // one arrival per MMA issuer
    }
    for (int g = 0; g < kQTiles; ++g) mbar_init(&bar_drain[g], 1);
    mbar_init(&bar_turn[0], 1);
    mbar_init(&bar_turn[1], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&take.full[s], 1);
      mbar_init(&take.empty[s], PAGED ? kUnitWalkers + 1 : kUnitWalkers);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort = &abort_flag;

  if (warp == 0 || (PAGED && warp == 3)) {
    regs_dec<kRegsControl>();
    // ================================================================ TMA producer(s)
    // Paged: warp 0 loads Q and the K tiles, warp 3 the V tiles. With 16-row pages a tile is 16
    // tensor boxes of 2 KB per 64-column block, more than one warp's lanes issue in time for
    // memory-bound batches (multi-token verify). Both walk every unit and every ring position.
    const bool v_warp = PAGED && warp == 3;
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
    }
    const uint64_t kv_policy = policy_evict_last();
    const uint64_t q_policy = policy_evict_first();
    uint32_t kv_it = 0;  // position in the K/V ring, continued across units
    Cursor cur = first_cursor<PAGED>(p, n_units);
    uint32_t requests = 0;  // launch cancellations requested
    for (int r = 0;; ++r) {
      const int u = next_unit<PAGED, TAKE>(p, cur, r, n_units, take, abort);
      if (u < 0) break;
      Unit w;
      unit_at<PAGED>(p, u, w);
      if (lane == 0 && !v_warp) {
        // the previous unit's last Q K^T must have read the Q tiles before they are replaced
        if (r > 0) mbar_wait(&bar_q_empty, (r - 1) & 1, abort, p.status, kSiteProducerEmpty);
        int n_active = 0;
#pragma unroll
        for (int g = 0; g < kQTiles; ++g) n_active += w.nkv[g] > 0;
        mbar_arrive_expect_tx(&bar_q_full, n_active * TB);
#pragma unroll
        for (int g = 0; g < kQTiles; ++g) {
          if (w.nkv[g] <= 0) continue;
          const int qrow = PAGED ? (int)(w.tok0 + w.row0[g] / p.pack) : w.row0[g];
          const int qbat = PAGED ? 0 : w.seq;
#pragma unroll
          for (int sub = 0; sub < C::kSub; ++sub)
            tma_load_4d_hint(sQ + g * TB + sub * C::kSubBytes, &p.tm_q, &bar_q_full, sub * 64, w.h, qrow, qbat,
                             q_policy);
        }
      }
      __syncwarp();
      // paged: page ids come 32 at a time, lane l holding the unit's page 32 b + l of batch b; the
      // next batch is read while the current one is used, so no page-table read is waited for
      // (past the keys the id is past the pool, where TMA reads zeros)
      const int ppt = PAGED ? kBN / p.page_size : 0;  // pages per key tile
      const int n_pages = w.nmax * ppt;                // pages of the unit's key range
      auto page_batch = [&](int b) {
        const int lp = w.kv_t0 * ppt + b * 32 + lane;  // logical page of this sequence
        return lp * p.page_size < w.kv_len ? p.page_table[(int64_t)w.seq * p.max_pages_per_seq + lp] : p.num_pages;
      };
      int pages_cur = 0, pages_next = 0, phys = 0;
      if (PAGED && n_pages > 0) pages_cur = page_batch(0);
      if (PAGED && n_pages > 32) pages_next = page_batch(1);
      for (int idx = 0; idx < 2 * w.nmax; ++idx, ++kv_it) {
        const int j = idx >> 1;
        const bool is_v = idx & 1;
        const int stage = kv_it % NS;
        if (PAGED && !is_v) {
          const int pj = j * ppt;  // the tile's first page within the unit
          if (j > 0 && (pj & 31) == 0) {
            pages_cur = pages_next;
            if (pj + 32 < n_pages) pages_next = page_batch((pj >> 5) + 1);
          }
          phys = __shfl_sync(0xffffffffu, pages_cur, (pj & 31) + (lane < ppt ? lane : 0));
        }
        if (PAGED && is_v != v_warp) continue;  // the other producer's stage
        if (lane == 0) mbar_wait(&bar_empty[stage], ((kv_it / NS) & 1) ^ 1, abort, p.status, kSiteProducerEmpty);
        __syncwarp();
        uint8_t* dst = sKV + stage * TB;
        const CUtensorMap* tm = is_v ? &p.tm_v : &p.tm_k;
        if (lane == 0) mbar_arrive_expect_tx(&bar_full[stage], TB);
        __syncwarp();
        if constexpr (!PAGED) {
          if (lane == 0) {
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub)
              tma_load_4d_hint(dst + sub * C::kSubBytes, tm, &bar_full[stage], sub * 64, w.hk, j * kBN, w.seq,
                               kv_policy);
          }
        } else {
          if (lane < ppt) {
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub)
              tma_load_4d_hint(dst + sub * C::kSubBytes + lane * p.page_size * 128, tm, &bar_full[stage],
                               sub * 64, w.hk, 0, phys, kv_policy);
          }
        }
        __syncwarp();
      }
      // The item's last unit is loaded: ask for the next item now, about a ring's depth of key
      // tiles before the walkers need it. One request is in flight at a time, and none follows a
      // failed one (the walk ends there).
      if (TAKE && cur.item_done() && !v_warp) {
        int issued = 0;
        if (lane == 0 && !*abort) {
          const uint32_t s = requests & 1;  // the slot's previous response must have been read
          if (requests < 2 || mbar_wait(&take.empty[s], ((requests >> 1) + 1) & 1, abort, p.status, kSiteTakeOver)) {
            fence_proxy_async_smem();  // the walkers' reads of the slot precede the new response
            mbar_arrive_expect_tx(&take.full[s], 16);
            launch_cancel_request(&take.resp[s], &take.full[s]);
            issued = 1;
          }
        }
        requests += __shfl_sync(0xffffffffu, issued, 0);
      }
    }
    // After an abort the walk may end before the last response arrived: wait for it (bounded)
    // so that nothing is written to this CTA's shared memory after it exits.
    if (TAKE && lane == 0 && *abort && requests > 0) {
      int no_abort = 0;
      mbar_wait(&take.full[(requests - 1) & 1], ((requests - 1) >> 1) & 1, &no_abort, p.status, kSiteTakeOver);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    regs_dec<kRegsControl>();
    // ================================================================ MMA issuers
    // Warp 1 issues every MMA of query tile 0, warp 2 those of query tile 1, taking turns (below).
    // With two issuers one warp's waits and commits overlap the other's MMA issue; a single issuer
    // serialises them and leaves the tensor core idle in between. Each K/V stage is released by
    // one commit from each issuer (its empty barrier counts two arrivals).
    const int g = warp - 1;
    const uint32_t idesc_s = make_idesc_bf16(kBM, kBN, false);
    const uint32_t idesc_pv = make_idesc_bf16(kBM, D, true);
    // Shared-memory descriptors are built once (see issue_qk / issue_pv for the K steps).
    // V is the MN-major B operand of P V: the two 64-column blocks of d sit 16 KB apart.
    const uint64_t dq = make_sdesc_sw128(smem_u32(sQ + g * TB), 16, 1024);
    const uint64_t dk = make_sdesc_sw128(smem_u32(sKV), 16, 1024);
    const uint64_t dv = make_sdesc_sw128(smem_u32(sKV), C::kSubBytes, 1024);
    const uint32_t tS = tmem + g * 128, tO = tmem + C::kColO + g * D;
    uint32_t kv_it = 0;   // ring position (K_j at kv_it + 2j, V_j at kv_it + 2j + 1)
    uint32_t tcnt = 0;    // key tiles of this query tile so far (bar_s / bar_p phases)
    uint32_t ounits = 0;  // units whose O this tile has produced (bar_o / bar_o_free phases)
    // The issuers take turns (0, 1, 0, 1, ...) and issue a step's MMAs only on their turn. That
    // keeps the tensor core's work in the order P0 V, Q0 K^T, P1 V, Q1 K^T, ...: one tile's
    // softmax runs while the tensor core serves the other tile. Without turns the two tiles drift
    // into lockstep, both softmaxes run at once and the tensor core idles meanwhile. Turns are
    // taken only at the steps where both tiles issue MMAs (the first Q K^T, then every key tile
    // both tiles attend to): both issuers know both tiles' key-tile counts, so they skip the same
    // steps. A unit with one query tile (decode, verify) then takes no turns at all. At d = 64
    // (separate P) the issuers take no turns: each issues a tile's next Q K^T as soon as its S has
    // been read and its P V as soon as P is written.
    uint32_t turn = 0;
    auto take_turn = [&]() {
      if (g == 0) {
        if (turn > 0) mbar_wait(&bar_turn[0], (turn - 1) & 1, abort, p.status, kSiteMmaTurn);
      } else {
        mbar_wait(&bar_turn[1], turn & 1, abort, p.status, kSiteMmaTurn);
      }
    };
    auto pass_turn = [&]() {
      mbar_arrive(&bar_turn[1 - g]);
      ++turn;
    };
    Cursor cur = first_cursor<PAGED>(p, n_units);
    for (int r = 0;; ++r) {
      const int u = next_unit<PAGED, TAKE>(p, cur, r, n_units, take, abort);
      if (u < 0) break;
      Unit w;
      unit_at<PAGED>(p, u, w);
      const int nkv = g == 0 ? w.nkv[0] : w.nkv[1];
      const int nkv_both = min(w.nkv[0], w.nkv[1]);  // key tiles at which both tiles issue MMAs
      if (lane == 0) {
        mbar_wait(&bar_q_full, r & 1, abort, p.status, kSiteMmaQ);
        if (nkv <= 0) mma_commit(&bar_q_empty);  // this tile reads no Q this unit
      }
      if (w.nmax > 0) {
        if (lane == 0) {
          const int ks0 = kv_it % NS;
          // Every issuer waits for a stage's fill before it arrives on the stage's empty barrier,
          // also when its tile does not read the stage: an issuer can then never arrive twice on
          // one pending phase, because the next fill waits for that phase to complete.
          mbar_wait(&bar_full[ks0], (kv_it / NS) & 1, abort, p.status, kSiteMmaFull);
          if (!kSepP && nkv_both > 0) take_turn();
          if (nkv > 0) {
            tc_fence_after();
            issue_qk<D>(tS, dq, dk + ks0 * (TB >> 4), idesc_s);
          }
          if (!kSepP && nkv_both > 0) pass_turn();
          if (nkv > 0) {
            mma_commit(&bar_s[g]);
            if (nkv == 1) mma_commit(&bar_q_empty);  // the unit's last Q K^T of this tile
          }
          mma_commit(&bar_empty[ks0]);
        }
        for (int j = 0; j < w.nmax; ++j) {
          const uint32_t vi = kv_it + 2 * j + 1, ki = kv_it + 2 * j + 2;
          const int vs = vi % NS, ks = ki % NS;
          const bool has_next = j + 1 < w.nmax;
          if constexpr (kSepP) {
            // the next key tile's Q K^T first: S is free once the softmax has read this tile's
            if (lane == 0 && has_next) {
              mbar_wait(&bar_full[ks], (ki / NS) & 1, abort, p.status, kSiteMmaFull);
              if (j + 1 < nkv) {
                mbar_wait(&bar_sfree[g], tcnt & 1, abort, p.status, kSiteMmaSFree);
                tc_fence_after();
                issue_qk<D>(tS, dq, dk + ks * (TB >> 4), idesc_s);
                mma_commit(&bar_s[g]);
                if (j + 2 == nkv) mma_commit(&bar_q_empty);  // the unit's last Q K^T of this tile
              }
              mma_commit(&bar_empty[ks]);
            }
            __syncwarp();
          }
          if (lane == 0) mbar_wait(&bar_full[vs], (vi / NS) & 1, abort, p.status, kSiteMmaFull);
          __syncwarp();
          if (j < nkv) {
            if constexpr (PAGED) {
              // Rows of the sequence's partial last page past kv_len hold no valid value (possibly
              // not even a finite one); P is 0 there but 0 * NaN is NaN, so they are zeroed first.
              // Both issuers write the same zeros, each before its own P V.
              const int t0 = (w.kv_t0 + j) * kBN;
              if (t0 < w.kv_len && w.kv_len < t0 + kBN && (w.kv_len % p.page_size) != 0) {
                const int r_begin = w.kv_len - t0;
                const int r_end = min(kBN, ((w.kv_len + p.page_size - 1) / p.page_size) * p.page_size - t0);
                uint8_t* vt = sKV + vs * TB;
                const int n_chunks = (r_end - r_begin) * C::kSub * 8;  // 16-byte chunks
                for (int c = lane; c < n_chunks; c += 32) {
                  const int row = r_begin + c / (C::kSub * 8);
                  const int sub = (c / 8) % C::kSub;
                  *reinterpret_cast<uint4*>(vt + sub * C::kSubBytes + row * 128 + (c & 7) * 16) =
                      make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
              }
              __syncwarp();
            }
            if (kSepP && lane == 0) {
              mbar_wait(&bar_p[g], tcnt & 1, abort, p.status, kSiteMmaP);
              // the first P V of a unit overwrites O: the previous unit's O must have been read
              if (j == 0 && ounits > 0) mbar_wait(&bar_o_free[g], (ounits - 1) & 1, abort, p.status, kSiteMmaP);
              tc_fence_after();
              issue_pv<D>(tO, tmem + kColP + g * 64, dv + vs * (TB >> 4), idesc_pv, j > 0 ? 1u : 0u);
              mma_commit(&bar_pv[g]);  // P and O are free for the next tile's softmax
              if (j == nkv - 1) {
                mma_commit(&bar_o[g]);
                ++ounits;
              }
            } else if (lane == 0) {
              mbar_wait(&bar_p[g], tcnt & 1, abort, p.status, kSiteMmaP);
              // the first P V of a unit overwrites O: the previous unit's O must have been read
              if (j == 0 && ounits > 0) mbar_wait(&bar_o_free[g], (ounits - 1) & 1, abort, p.status, kSiteMmaP);
              if (j + 1 < nkv) mbar_wait(&bar_full[ks], (ki / NS) & 1, abort, p.status, kSiteMmaFull);
              if (j < nkv_both) take_turn();
              tc_fence_after();
              issue_pv<D>(tO, tS, dv + vs * (TB >> 4), idesc_pv, j > 0 ? 1u : 0u);
              if (j + 1 < nkv) issue_qk<D>(tS, dq, dk + ks * (TB >> 4), idesc_s);
              if (j < nkv_both) pass_turn();
              if (j == nkv - 1) {
                mma_commit(&bar_o[g]);
                ++ounits;
              }
              if (j + 1 < nkv) {
                mma_commit(&bar_s[g]);
                if (j + 2 == nkv) mma_commit(&bar_q_empty);  // the unit's last Q K^T of this tile
              }
            }
            ++tcnt;
          }
          if (lane == 0) {
            mma_commit(&bar_empty[vs]);
            if (!kSepP && has_next) {
              if (j + 1 >= nkv) mbar_wait(&bar_full[ks], (ki / NS) & 1, abort, p.status, kSiteMmaFull);
              mma_commit(&bar_empty[ks]);
            }
          }
          __syncwarp();
        }
        kv_it += 2 * w.nmax;
      }
      __syncwarp();
    }
    // drain: every MMA this warp issued has completed before TMEM is released
    if (lane == 0) {
      mma_commit(&bar_drain[g]);
      int no_abort = 0;
      mbar_wait(&bar_drain[g], 0, &no_abort, p.status, kSiteDrain);
    }
    __syncwarp();
  } else if (warp == 3) {
    regs_dec<kRegsControl>();  // dense layout: idle
  } else if (warp >= 4) {
    regs_inc<kRegsSoftmax>();
    // ================================================================ softmax warpgroups
    const int g = (warp - 4) >> 2;
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int r_in = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + g * 128 + lane_off;
    const uint32_t tO = tmem + C::kColO + g * D + lane_off;
    const float sl2 = p.scale_log2;
    uint32_t tcnt = 0, ounits = 0;
    Cursor cur = first_cursor<PAGED>(p, n_units);
    for (int r = 0;; ++r) {
      const int u = next_unit<PAGED, TAKE>(p, cur, r, n_units, take, abort);
      if (u < 0) break;
      Unit w;
      unit_at<PAGED>(p, u, w);
      const int nkv = g == 0 ? w.nkv[0] : w.nkv[1];
      if (nkv < 0) continue;
      const int prow = (g == 0 ? w.row0[0] : w.row0[1]) + r_in;  // packed row of this thread
      const int pack = PAGED ? p.pack : 1;
      const int row = prow / pack;                                   // query token in the sequence
      const int head = w.h + prow % pack;
      const int lim_row = p.causal ? min(w.kv_len, row + w.off + 1) : w.kv_len;  // keys [0, lim_row)
      // A warp none of whose rows is a query row of the unit (the padding of a packed tile with
      // few tokens) keeps every barrier phase but does no work: MMA rows are independent, and
      // its rows' P and O are never stored.
      const bool live = __any_sync(0xffffffffu, row < w.q_len);
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkv; ++j, ++tcnt) {
        mbar_wait(&bar_s[g], tcnt & 1, abort, p.status, kSiteSoftmaxS);
        __syncwarp();  // lanes leave the wait at different times; tcgen05.ld is warp-collective
        if (!live) {
          if constexpr (kSepP) {
            mbar_arrive(&bar_sfree[g]);
            // The next S can be ready before the live warps release this tile's P; arriving on
            // bar_p only once the previous tile's P V is done keeps this warp's arrivals in the
            // phase of the tile they belong to.
            if (j > 0) mbar_wait(&bar_pv[g], (tcnt - 1) & 1, abort, p.status, kSiteSoftmaxPV);
          }
          mbar_arrive(&bar_p[g]);
          continue;
        }
        tc_fence_after();
        const int valid = lim_row - (w.kv_t0 + j) * kBN;
        if (__any_sync(0xffffffffu, valid < kBN)) {
          // Tiles that cross the diagonal or the end of the keys: the masked scores are set to
          // -inf in TMEM, one 32-column chunk at a time in a loop that is not unrolled, so that
          // this rarely taken path adds little code to the loop every tile runs.
#pragma unroll 1
          for (int cc = 0; cc < kBN / 32; ++cc) {
            uint32_t mr[32];
            tmem_ld32(tS + cc * 32, mr);
            tmem_ld_wait(mr);
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (cc * 32 + c >= valid) mr[c] = 0xff800000u;  // -inf
            tmem_st32(tS + cc * 32, mr);
          }
          tmem_st_wait();
        }
        uint32_t sr[kBN];
        tmem_ld32(tS + 0, sr + 0);
        tmem_ld32(tS + 32, sr + 32);
        tmem_ld32(tS + 64, sr + 64);
        tmem_ld32(tS + 96, sr + 96);
        tmem_ld_wait(sr + 0);
        tmem_ld_wait(sr + 32);
        tmem_ld_wait(sr + 64);
        tmem_ld_wait(sr + 96);
        if constexpr (kSepP) {
          tc_fence_before();
          mbar_arrive(&bar_sfree[g]);  // S is in registers: the next tile's Q K^T may overwrite it
        }
        const float m_tile = row_max_chunks<0, 4>(sr) * sl2;
        const bool need = m_tile > m_run + kRescaleThreshold;
        const float alpha = need ? ex2(m_run - m_tile) : 1.f;  // 0 while m_run is -inf
        if (need) m_run = m_tile;
        const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
        float la, lb;
        if constexpr (kSepP) {
          uint32_t pk[kBN / 2];
          split_f32x2(softmax_regs(sr, sl2, neg_m, pk), la, lb);
          if (j > 0) {
            // the previous tile's P V must have read P and written O
            mbar_wait(&bar_pv[g], (tcnt - 1) & 1, abort, p.status, kSiteSoftmaxPV);
            __syncwarp();
            tc_fence_after();
          }
          rescale_o<D>(tO, j > 0 && __any_sync(0xffffffffu, need), alpha);
          const uint32_t tP = tmem + kColP + g * 64 + lane_off;
#pragma unroll
          for (int cc = 0; cc < kBN / 32; ++cc) tmem_st16(tP + cc * 16, pk + cc * 16);
        } else {
          split_f32x2(softmax_chunks<0, 4>(sr, sl2, neg_m, tS), la, lb);
          // after P is written, so S no longer occupies registers
          rescale_o<D>(tO, j > 0 && __any_sync(0xffffffffu, need), alpha);
        }
        l_run = fmaf(l_run, alpha, la + lb);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_p[g]);
        __syncwarp();
      }
      // ------------------------------------------------------------ epilogue: O / l, LSE
      // O is read from TMEM and stored one 32-column chunk at a time, in a loop that is not
      // unrolled (this code runs once per unit; small code keeps the per-tile loop in the
      // instruction cache). The MMA may overwrite O once every chunk has been read.
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const int64_t tok = w.tok0 + row;
      const bool store = row < w.q_len && (!PAGED || tok < p.total_q);
      // a split unit writes its fp32 partial state into its split's part
      float* o_f32 = p.o_f32;
      float* lse_out = p.lse;
      int64_t orow = tok * p.Hq + head;
      if (PAGED && p.kv_splits > 1) {
        o_f32 = p.o_part;
        lse_out = p.lse_part;
        orow += (int64_t)w.split * p.total_q * p.Hq;
      }
      if (nkv > 0) {
        mbar_wait(&bar_o[g], ounits & 1, abort, p.status, kSiteSoftmaxO);
        __syncwarp();
        ++ounits;
        if (!live) {
          mbar_arrive(&bar_o_free[g]);
          continue;
        }
        tc_fence_after();
      }
      const uint64_t il2 = f32x2(inv_l, inv_l);
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t orr[32];
        if (nkv > 0) {
          tmem_ld32(tO + cc * 32, orr);
          tmem_ld_wait(orr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = 0u;
        }
        float on[32];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          split_f32x2(mul_f32x2(f32x2(u2f(orr[2 * i]), u2f(orr[2 * i + 1])), il2), on[2 * i], on[2 * i + 1]);
        if (store && o_f32 != nullptr) {
          float4* dst = reinterpret_cast<float4*>(o_f32 + orow * D + cc * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(on[4 * i], on[4 * i + 1], on[4 * i + 2], on[4 * i + 3]);
        } else if (store) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + orow * D + cc * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack_bf16x2(on[8 * i + 0], on[8 * i + 1]), pack_bf16x2(on[8 * i + 2], on[8 * i + 3]),
                                pack_bf16x2(on[8 * i + 4], on[8 * i + 5]), pack_bf16x2(on[8 * i + 6], on[8 * i + 7]));
        }
      }
      if (nkv > 0) {
        tc_fence_before();
        mbar_arrive(&bar_o_free[g]);  // the MMA may now overwrite O with the next unit
      }
      if (store && lse_out != nullptr) lse_out[orow] = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Work list for the paged prefill: one item per (sequence, pair of query tiles). Sequences come
// longest first (a stable counting sort on their key-tile count); the items of one sequence are
// contiguous, heaviest query tiles first, so the CTAs running together share one sequence's K/V
// pages in L2 while the order still starts with the longest work. One CTA does it, in parallel:
// with at most one sequence per thread each thread counts the sequences that sort before its own;
// larger batches take a histogram of the counts, a scan of the buckets (longest first), a stable
// placement in chunks of one sequence per thread (warps of a chunk in turn, so equal counts keep
// their index order), and a scan of the item counts in the sorted order.
constexpr int kPlanThreads = 1024;

// Exclusive scan across the block of one int per thread; returns this thread's prefix and leaves
// the block total in *total_out. Uses warp_sums[32] of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total_out) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive scan of the warp totals
  }
  __syncthreads();
  const int excl = incl - v + (wid > 0 ? warp_sums[wid - 1] : 0);
  *total_out = warp_sums[nw - 1];
  __syncthreads();  // warp_sums may be reused by the next scan
  return excl;
}

__global__ void __launch_bounds__(kPlanThreads) plan_paged_kernel(
    const int32_t* __restrict__ cu, const int32_t* __restrict__ kv_lens, int num_seqs, int causal, int pack,
    int max_cost, int max_items, int2* __restrict__ work_list, int* __restrict__ work_count,
    int* __restrict__ scratch) {
  extern __shared__ int plan_smem[];  // max_cost + 1 buckets, or (<= nt sequences) 2 * nt ints
  __shared__ int warp_sums[32];
  // the key-row decode kernel after this one may start its set-up now (it waits for this kernel's
  // results before reading them)
  if (threadIdx.x == 0) griddep_launch_dependents();
  __shared__ int total;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, wid = tid >> 5;
  auto cost_in = [&](int s) {
    const int kv = kv_lens[s];
    return min(kv > 0 ? (kv + kBN - 1) / kBN : 0, max_cost);
  };
  auto items_in = [&](int s) {
    const int q_len = cu[s + 1] - cu[s];
    return q_len > 0 ? (q_len * pack + 2 * kBM - 1) / (2 * kBM) : 0;
  };
  // order[k]: the k-th sequence of the sorted order
  int* order = num_seqs <= nt ? plan_smem + nt : scratch;
  if (num_seqs <= nt) {
    // one sequence per thread: rank = sequences that sort before this one
    int* s_cost = plan_smem;
    const int my_cost = tid < num_seqs ? cost_in(tid) : -1;
    if (tid < num_seqs) s_cost[tid] = my_cost;
    __syncthreads();
    if (tid < num_seqs) {
      int rank = 0;
      for (int j = 0; j < num_seqs; ++j) {
        const int c = s_cost[j];
        rank += (c > my_cost) | ((c == my_cost) & (j < tid));
      }
      order[rank] = tid;
    }
    __syncthreads();
  } else {
    int* hist = plan_smem;  // per count: sequences, then the next free position of that count
    for (int c = tid; c <= max_cost; c += nt) hist[c] = 0;
    __syncthreads();
    for (int s = tid; s < num_seqs; s += nt) atomicAdd(&hist[cost_in(s)], 1);
    __syncthreads();
    // bucket starts, longest first: each thread scans a run of counts from the top down
    const int per = (max_cost + 1 + nt - 1) / nt;
    const int hi = max_cost - tid * per;  // this thread's counts: hi, hi-1, ..., hi-per+1 (>= 0)
    int mine = 0;
    for (int i = 0; i < per; ++i)
      if (hi - i >= 0) mine += hist[hi - i];
    int unused;
    int run = block_exclusive_scan(mine, warp_sums, &unused);
    for (int i = 0; i < per; ++i)
      if (hi - i >= 0) {
        const int t = hist[hi - i];
        hist[hi - i] = run;
        run += t;
      }
    __syncthreads();
    // stable placement, one chunk of nt sequences at a time, the warps of a chunk in turn
    for (int base = 0; base < num_seqs; base += nt) {
      const int s = base + tid;
      const int c = s < num_seqs ? cost_in(s) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, c);
      const int leader = __ffs(peers) - 1;
      const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
      for (int w = 0; w < nt / 32; ++w) {
        if (wid == w && s < num_seqs && lane == leader) {
          const int start = hist[c];
          hist[c] = start + __popc(peers);
          warp_sums[lane] = start;  // handed to the group below
        }
        __syncwarp();
        if (wid == w && s < num_seqs) order[warp_sums[leader] + rank_in_warp] = s;
        __syncthreads();
      }
    }
  }
  // item offsets in the sorted order: each thread scans a run of consecutive positions
  const int per = (num_seqs + nt - 1) / nt;
  const int k0 = tid * per;
  int mine = 0;
  for (int i = 0; i < per && k0 + i < num_seqs; ++i) mine += items_in(order[k0 + i]);
  int all_items;
  int run = block_exclusive_scan(mine, warp_sums, &all_items);
  if (tid == 0) {
    total = min(all_items, max_items);  // more items than the host bound means inconsistent lengths
    work_count[0] = total;
    work_count[1] = 0;  // the unit counter of the decode kernel's persistent CTAs
  }
  __syncthreads();
  for (int i = 0; i < per && k0 + i < num_seqs; ++i) {
    const int s = order[k0 + i];
    const int n = items_in(s);
    for (int it = 0; it < n; ++it) {
      const int pos = run + it;
      if (pos < total) work_list[pos] = make_int2(s, causal ? n - 1 - it : it);
    }
    run += n;
  }
}

// Grid size: one CTA per work item — dense causal, two mirrored query-tile pairs (item_unit);
// otherwise one unit — and a CTA that finishes takes over a pending CTA's item (next_unit)
// instead of exiting. Items then run in the hardware's launch order, the order the units are
// numbered in for L2 reuse, which measured faster than a persistent grid with a static order.
// FA_PREFILL_TAKE_OVER=0 turns the take-over off: dense CTAs then exit after their own item and
// paged work runs on a persistent grid (one CTA per SM, snake order). FA_PREFILL_PERSISTENT=0
// (one CTA per unit, no take-over) or 1 (persistent) overrides both.
int env_mode(const char* name) {
  const char* e = getenv(name);
  return (e == nullptr || (e[0] != '0' && e[0] != '1')) ? -1 : (e[0] == '1');  // -1: not set
}
int persistent_override() {
  static const int mode = env_mode("FA_PREFILL_PERSISTENT");
  return mode;
}
int take_over_enabled() {
  static const int mode = env_mode("FA_PREFILL_TAKE_OVER");
  return mode != 0;
}

template <int D, bool PAGED, bool TAKE = false>
cudaError_t launch_prefill_impl(const PrefillParams& p, int grid, cudaStream_t stream) {
  auto kern = prefill_kernel<D, PAGED, TAKE>;
  {
    // The register split (kRegsControl / kRegsSoftmax) draws on the registers the CTA launches
    // with; a larger split would make the increase wait forever, so refuse to launch instead.
    // (The caches below are atomics: calls may come from several host threads at once.)
    static std::atomic<int> launch_regs{-1};
    int regs = launch_regs.load(std::memory_order_relaxed);
    if (regs < 0) {
      cudaFuncAttributes attr;
      const cudaError_t e = cudaFuncGetAttributes(&attr, kern);
      if (e != cudaSuccess) return e;
      regs = attr.numRegs;
      launch_regs.store(regs, std::memory_order_relaxed);
    }
    if (128 * kRegsControl + 256 * kRegsSoftmax > kPrefillThreads * regs) return cudaErrorInvalidConfiguration;
  }
  static std::atomic<unsigned> configured_mask{0u};  // one bit per device ordinal below 32
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 32 || !(configured_mask.load(std::memory_order_acquire) & (1u << dev))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 32) configured_mask.fetch_or(1u << dev, std::memory_order_release);
  }
  kern<<<grid, kPrefillThreads, Cfg<D>::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_dense(const PrefillParams& p, int d, int sm_count, cudaStream_t stream) {
  const int n2 = (p.S + 2 * kBM - 1) / (2 * kBM);
  const long long units = (long long)n2 * p.B * p.Hq;
  const int mode = persistent_override();
  PrefillParams q = p;
  int grid;
  bool take = false;
  if (mode == 1) {
    grid = (int)(units < sm_count ? units : sm_count);
  } else if (mode == 0 || !p.causal) {
    grid = (int)units;
    take = mode != 0 && take_over_enabled();
  } else {
    q.pair_units = 1;  // causal: mirrored query-tile pairs, one pair per work item
    take = take_over_enabled();
    grid = ((n2 + 1) / 2) * p.B * p.Hq;
  }
  if (d == 128) {
    return take ? launch_prefill_impl<128, false, true>(q, grid, stream) : launch_prefill_impl<128, false>(q, grid, stream);
  }
  return take ? launch_prefill_impl<64, false, true>(q, grid, stream) : launch_prefill_impl<64, false>(q, grid, stream);
}

cudaError_t launch_plan_paged(const PrefillParams& p, int max_items, int max_kv_tiles, int2* work_list,
                              int* work_count, cudaStream_t stream) {
  // buckets (at most 8193 ints), or for batches of at most one sequence per thread their counts
  // and order (2 x 1024 ints): within the default dynamic shared memory limit either way
  const int smem = (p.num_seqs <= kPlanThreads ? 2 * kPlanThreads : max_kv_tiles + 1) * (int)sizeof(int);
  int* scratch = reinterpret_cast<int*>(work_list + max_items);  // 2 * num_seqs ints
  plan_paged_kernel<<<1, kPlanThreads, smem, stream>>>(p.cu_seqlens_q, p.kv_lens, p.num_seqs, p.causal, p.pack,
                                                       max_kv_tiles, max_items, work_list, work_count, scratch);
  return cudaGetLastError();
}

cudaError_t launch_prefill_paged(const PrefillParams& p, int d, int sm_count, int max_items, int max_kv_tiles,
                                 int2* work_list, int* work_count, cudaStream_t stream, cudaEvent_t after_plan) {
  cudaError_t e = launch_plan_paged(p, max_items, max_kv_tiles, work_list, work_count, stream);
  if (e == cudaSuccess && after_plan != nullptr) e = cudaEventRecord(after_plan, stream);
  if (e != cudaSuccess) return e;
  const long long units = (long long)max_items * (p.Hq / p.pack) * p.kv_splits;
  const int mode = persistent_override();
  const bool take = mode == -1 && take_over_enabled();
  const bool persistent = mode == 1 || (mode == -1 && !take);
  const int grid = (int)((units < sm_count || !persistent) ? units : sm_count);
  if (d == 128) {
    return take ? launch_prefill_impl<128, true, true>(p, grid, stream) : launch_prefill_impl<128, true>(p, grid, stream);
  }
  return take ? launch_prefill_impl<64, true, true>(p, grid, stream) : launch_prefill_impl<64, true>(p, grid, stream);
}

}  // namespace fa
