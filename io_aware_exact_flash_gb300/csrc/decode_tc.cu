// Tensor-core decode and verify over a paged KV cache with the keys on the MMA's row dimension.
//
// Decoding attends a few query rows per (sequence, kv head) — one token times the GQA group, or a
// handful of tokens for multi-token verify — to the sequence's whole key set, read through its
// page table ("I/O-Aware Kernels", datasystem.school Module 5, section "FlashInfer: I/O-aware
// attention for serving"). The work is a stream over the cache, bound by reading K and V once;
// the online softmax of the section "FlashAttention: tiling + online softmax" keeps every score
// on chip. Put on the tensor cores the usual way (query rows as the MMA's M = 128 rows), a tile
// holds only a handful of real rows and each key tile costs a full 128-row Q K^T, softmax and P V
// chain in series. Here the roles are swapped: a key tile of 128 keys is the MMA's M dimension
// and the query rows are its N = 16 columns:
//   S^T[128 keys, N] = K_tile [128, d] . Q^T           (tcgen05.mma, A = K, B = Q, both K-major)
//   O^T[d, N]       += V_tile^T [d, 128 keys] . P^T    (A = V read MN-major, B = P^T K-major)
// so each MMA is small, one softmax thread owns one key (one TMEM lane), and the chain per key tile
// is short next to the time its 64 KB take to arrive: the kernel runs at the pace of HBM.
//
// The softmax runs per query column with a running maximum m that is raised only when a score
// exceeds it by more than 2^8. Each tile, the four softmax warps vote (through shared memory)
// whether any score does; only then are the column maxima gathered (a warp reduction, then the
// four warps' values) and m, the partial sums and O^T's columns rescaled. Each thread keeps a
// partial row sum l over its key rows, summed across the 128 threads once per unit. P^T is written to shared memory as bf16 in the
// MMA's swizzled K-major layout.
//
// A unit is (sequence, kv head, key split). The CTAs are persistent (one per SM) and take units in
// the planner's order (longest sequences first) from a counter in global memory; a scheduler warp
// claims the next unit and reads its first 32 page ids while the TMA warp issues the current unit's
// last loads, so the TMA warp streams straight from one unit's keys into the next and a CTA never
// holds a unit it has not started while others run out of work. Split units write fp32 partial states merged afterwards by
// their LSE (merge_kernel).
//
// CTA organisation (288 threads):
//   warps 0, 2  TMA producers: per unit its Q rows (warp 0), then K_0, V_0, K_1, V_1, ... into a
//               stage ring, the K tiles from warp 0 and the V tiles from warp 2 (with 16-row pages a
//               tile is 16 tensor boxes of 2 KB, and one warp's lanes cannot issue them fast enough
//               to keep up with HBM)
//   warp 1      S^T issuer (one lane): S^T of key tile j as soon as its keys are in and its buffer
//               is free (S^T is double buffered, so it runs during the previous tile's softmax)
//   warp 4      P V issuer (one lane): O^T += V^T P^T once the tile's P^T is written. Each
//               tcgen05.mma issue takes ~100 cycles however small the MMA, so the two streams of
//               eight MMAs per tile are issued by two warps side by side.
//   warp 2      also TMEM owner
//   warp 3      unit scheduler
//   warps 5-8   softmax: thread i owns key row i of each tile (TMEM lane i, its warp's lane
//               quarter) and, in the epilogue, row d = i of O^T
// TMEM columns: S^T buffers at [0, N) and [N, 2N), O^T buffers (one per unit parity) at [2N, 3N)
// and [3N, 4N).
#include <cuda_bf16.h>
#include <atomic>
#include "kernels.cuh"

namespace fa {

namespace {

constexpr int kKeys = 128;                        // keys per tile: TMEM lanes of S^T, rows of a stage
constexpr int kHd = 128;                          // head dim served by this kernel
constexpr int kStageBytes = kKeys * kHd * 2;      // one K or V tile (bf16): 32 KB
constexpr int kBlockBytes = kKeys * 128;          // one 64-column block of a stage: 16 KB
constexpr int kUnitSlots = 4;                     // units the scheduler may run ahead
constexpr float kKrRescaleThreshold = 8.0f;       // log2 units: 2^8, as in the prefill kernel
constexpr float kKrLn2 = 0.6931471805599453f;

// Wait sites recorded in the device status word when a wait times out.
enum : uint32_t {
  kSiteKrUnit = 32,
  kSiteKrQ = 33,
  kSiteKrFull = 34,
  kSiteKrEmpty = 35,
  kSiteKrS = 36,
  kSiteKrSFree = 37,
  kSiteKrP = 38,
  kSiteKrPFree = 39,
  kSiteKrO = 40,
  kSiteKrOFree = 41,
  kSiteKrX = 42,
  kSiteKrDrain = 43,
};

template <int N>
struct KrCfg {
  static_assert(N == 16, "query columns per unit: 16");
  static constexpr int kRowBytes = N * 128;                  // one 64-column block of N rows
  static constexpr int kQBytes = 2 * kRowBytes;              // Q: N rows x 128 (two blocks)
  static constexpr int kPBytes = 2 * kRowBytes;              // P^T: N rows x 128 keys (two blocks)
  // Six 32 KB stages. The count must be even: K_j sits at ring position 2j and V_j at 2j + 1, so with an even count
  // the K tiles only ever use the even stages and the V tiles the odd ones, and each stage has a
  // single producer (warp 0 or 2) and a single consumer (the S^T or the P V issuer) taking its
  // positions in order. With an odd count a stage would carry K and V tiles in turn, and the S^T
  // issuer, which runs ahead of the P V stream, could take a phase of a stage's full barrier that
  // belongs to a V tile not yet landed (parity waits tell phases apart only one phase deep).
  static constexpr int kStages = 6;
  static_assert(kStages % 2 == 0, "K and V tiles must not share ring stages");
  static constexpr int kSmemBytes = 1024 + 2 * kQBytes + 2 * kPBytes + kStages * kStageBytes;
  static constexpr uint32_t kTmemCols = 4 * N;               // 64 or 128: a power of two >= 32
};

// A unit as the scheduler publishes it. end = 1: no more units.
struct KrUnit {
  int end, seq, hk, split, ntiles, kv_t0, kv_len, q_len;
  long long tok0;  // first query row of the sequence
};

// R consecutive TMEM columns (R = 4, 8, 16 or 32) of this warp's 32 lanes into r, waited for.
template <int R>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  if constexpr (R == 32) {
    tmem_ld32(taddr, r);
    tmem_ld_wait(r);
  } else if constexpr (R == 16) {
    tmem_ld16(taddr, r);
    tmem_ld_wait16(r);
  } else if constexpr (R == 8) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr)
        : "memory");
  } else {
    static_assert(R == 4, "4, 8, 16 or 32 columns");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(taddr)
        : "memory");
  }
}
template <int R>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t* r) {
  if constexpr (R == 32) {
    tmem_st32(taddr, r);
  } else if constexpr (R == 16) {
    tmem_st16(taddr, r);
  } else if constexpr (R == 8) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]));
  } else {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3]));
  }
}

// Start-address step (16-byte units) of K step kk (16 elements) in a 128-byte-swizzled K-major
// operand whose 64-column blocks are block_bytes apart: 32 bytes inside a swizzle row, the next
// block every four steps.
__device__ __forceinline__ uint64_t kmajor_step(int kk, int block_bytes) {
  return (uint64_t)((kk >> 2) * (block_bytes >> 4) + (kk & 3) * 2);
}

// N: query columns of the MMAs (16); R: columns the softmax computes (4, 8 or 16; at least every
// unit's q_len x group). Columns at or past a unit's rows are masked like keys past
// its end, so the softmax loops have a compile-time trip count and no per-column branches.
template <int N, int R>
__global__ void __launch_bounds__(288, 1) decode_tc_kernel(const __grid_constant__ PrefillParams p) {
  static_assert(R <= N, "softmax columns within the MMA's columns");
  using C = KrCfg<N>;
  constexpr int NS = C::kStages;

  extern __shared__ uint8_t kr_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(kr_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                    // two Q buffers (unit parity)
  uint8_t* sP = sQ + 2 * C::kQBytes;     // two P^T buffers (tile parity)
  uint8_t* sKV = sP + 2 * C::kPBytes;    // NS stages

  __shared__ uint64_t bar_full[NS], bar_empty[NS];
  __shared__ uint64_t bar_q_full[2], bar_q_empty[2];
  __shared__ uint64_t bar_s_full[2], bar_s_free[2], bar_p_full[2], bar_p_free[2];
  __shared__ uint64_t bar_o_full[2], bar_o_free[2];
  __shared__ uint64_t bar_x[2];  // the softmax warps' exchanges, two phases in turn
  __shared__ uint64_t bar_u_full[kUnitSlots], bar_u_empty[kUnitSlots];
  __shared__ uint64_t bar_drain[2];
  __shared__ uint64_t bar_req;  // the producer asks for the next unit
  __shared__ KrUnit units[kUnitSlots];
  __shared__ int unit_pages[kUnitSlots][32];  // physical ids of a unit's first 32 pages
  __shared__ alignas(16) float xred[2][N][4];  // per column, the four softmax warps' values
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // a key-split merge after this kernel may be made resident now; it waits for this kernel
    griddep_launch_dependents();
    abort_flag = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_q_full[b], 1);
      mbar_init(&bar_q_empty[b], 1);
      mbar_init(&bar_s_full[b], 1);
      mbar_init(&bar_s_free[b], 128);
      mbar_init(&bar_p_full[b], 128);
      mbar_init(&bar_p_free[b], 1);
      mbar_init(&bar_o_full[b], 1);
      mbar_init(&bar_o_free[b], 128);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&bar_x[b], 4);
    for (int s = 0; s < kUnitSlots; ++s) {
      mbar_init(&bar_u_full[s], 1);
      mbar_init(&bar_u_empty[s], 8);  // two producers, two issuers, four softmax warps
    }
    mbar_init(&bar_drain[0], 1);
    mbar_init(&bar_drain[1], 1);
    mbar_init(&bar_req, 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // launched while the planning kernel may still run: its work list and unit counter (and so
  // everything after this point) wait for it to finish
  griddep_wait();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort = &abort_flag;
  const int G = p.group;

  // Every consumer of the unit ring: wait for slot r, copy the unit, release the slot. Returns
  // false at the end of the work or after an abort (the slot is then not used).
  auto take_unit = [&](int r, KrUnit& x, int* page0 = nullptr) -> bool {
    const int slot = r % kUnitSlots;
    bool ok = true;
    if (lane == 0) ok = mbar_wait(&bar_u_full[slot], (r / kUnitSlots) & 1, abort, p.status, kSiteKrUnit);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok || *abort) return false;
    x = units[slot];
    if (page0 != nullptr) *page0 = unit_pages[slot][lane];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar_u_empty[slot]);
    return x.end == 0;
  };

  if (warp == 3) {
    // ================================================================ unit scheduler
    const int S = p.kv_splits;
    const int n_units = *p.work_count * p.Hkv * S;
    int* counter = const_cast<int*>(p.work_count) + 1;  // zeroed by the planning kernel
    const int ppt = kKeys / p.page_size;                 // pages per key tile (1..8)
    for (int r = 0;; ++r) {
      const int slot = r % kUnitSlots;
      if (lane == 0) {
        // Unit r is claimed only when the producer asks for it, near the end of unit r - 1's loads:
        // claimed earlier, a long unit in progress would hold it while other CTAs run out of work.
        if (r >= 1) mbar_wait(&bar_req, (r - 1) & 1, abort, p.status, kSiteKrUnit);
        if (r >= kUnitSlots) mbar_wait(&bar_u_empty[slot], ((r / kUnitSlots) - 1) & 1, abort, p.status, kSiteKrUnit);
      }
      __syncwarp();
      int u = 0;
      if (lane == 0) u = atomicAdd(counter, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      KrUnit& x = units[slot];
      if (u >= n_units || *abort) {
        if (lane == 0) {
          x.end = 1;
          mbar_arrive(&bar_u_full[slot]);
        }
        break;
      }
      const int item = u / (p.Hkv * S), rem = u - item * (p.Hkv * S);
      const int hk = rem / S, split = rem - hk * S;
      const int seq = p.work_list[item].x;
      const int c0 = p.cu_seqlens_q[seq], c1 = p.cu_seqlens_q[seq + 1];
      const int kv_len = min(p.kv_lens[seq], p.max_pages_per_seq * p.page_size);
      const int nkv = kv_len > 0 ? (kv_len + kKeys - 1) / kKeys : 0;
      const int per = (nkv + S - 1) / S;  // split s takes key tiles [s per, (s + 1) per)
      const int kv_t0 = split * per;
      const int ntiles = max(0, min(nkv - kv_t0, per));
      {
        const int lp = kv_t0 * ppt + lane;
        unit_pages[slot][lane] = (ntiles > 0 && lp * p.page_size < kv_len)
                                     ? p.page_table[(int64_t)seq * p.max_pages_per_seq + lp]
                                     : p.num_pages;  // past the pool: TMA fills zeros
      }
      if (lane == 0) {
        x.end = 0;
        x.seq = seq;
        x.hk = hk;
        x.split = split;
        x.ntiles = ntiles;
        x.kv_t0 = kv_t0;
        x.kv_len = kv_len;
        x.q_len = c1 - c0;
        x.tok0 = c0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_u_full[slot]);
    }
  } else if (warp == 0 || warp == 2) {
    // ================================================================ TMA producers
    // Both walk every unit and the whole ring; warp 0 loads Q and the K stages, warp 2 the V stages.
    const bool v_warp = warp == 2;
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
    }
    const uint64_t policy = policy_evict_first();  // every K/V and Q byte is read once
    const int ppt = kKeys / p.page_size;
    const int q_rows = (N / G) * G;  // rows of the Q box: whole tokens of the group's heads
    uint32_t kv_it = 0;
    for (int r = 0;; ++r) {
      KrUnit x;
      // Page ids come 32 at a time, lane l holding the unit's page 32 b + l of batch b: the next
      // batch is read while the current one is used, so no page-table read is ever waited for.
      int pages_cur = 0, pages_next = 0;
      if (!take_unit(r, x, &pages_cur)) break;
      const int qb = r & 1;
      if (lane == 0 && !v_warp) {
        if (r >= 2) mbar_wait(&bar_q_empty[qb], ((r >> 1) - 1) & 1, abort, p.status, kSiteKrQ);
        mbar_arrive_expect_tx(&bar_q_full[qb], 2 * q_rows * 128);
#pragma unroll
        for (int sub = 0; sub < 2; ++sub)
          tma_load_4d_hint(sQ + qb * C::kQBytes + sub * C::kRowBytes, &p.tm_q, &bar_q_full[qb], sub * 64, x.hk * G,
                           (int)x.tok0, 0, policy);
      }
      __syncwarp();
      const int n_pages = x.ntiles * ppt;  // pages of this unit
      auto page_batch = [&](int b) {
        const int lp = x.kv_t0 * ppt + b * 32 + lane;
        return lp * p.page_size < x.kv_len ? p.page_table[(int64_t)x.seq * p.max_pages_per_seq + lp] : p.num_pages;
      };
      if (n_pages > 32) pages_next = page_batch(1);
      int phys = 0;  // lane l < ppt: physical id of page l of the current key tile
      // ask for the next unit when the K tile before this unit's last one is loaded (at once for a
      // unit of at most two key tiles): its fetch then overlaps the ring's last tiles of this one
      const int req_idx = x.ntiles >= 2 ? 2 * (x.ntiles - 2) : 0;
      if (lane == 0 && x.ntiles == 0 && !v_warp) mbar_arrive(&bar_req);
      for (int idx = 0; idx < 2 * x.ntiles; ++idx, ++kv_it) {
        const int j = idx >> 1;
        const bool is_v = idx & 1;
        const int stage = kv_it % NS;
        if (lane == 0 && idx == req_idx && !v_warp) mbar_arrive(&bar_req);
        if (!is_v) {
          const int pj = j * ppt;  // the tile's first page within the unit
          if (j > 0 && (pj & 31) == 0) {
            pages_cur = pages_next;
            if (pj + 32 < n_pages) pages_next = page_batch((pj >> 5) + 1);
          }
          phys = __shfl_sync(0xffffffffu, pages_cur, (pj & 31) + (lane < ppt ? lane : 0));
        }
        if (is_v != v_warp) continue;  // the other producer's stage
        if (lane == 0) mbar_wait(&bar_empty[stage], ((kv_it / NS) & 1) ^ 1, abort, p.status, kSiteKrEmpty);
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&bar_full[stage], kStageBytes);
        __syncwarp();
        if (lane < ppt) {
          uint8_t* dst = sKV + stage * kStageBytes + lane * p.page_size * 128;
          const CUtensorMap* tm = is_v ? &p.tm_v : &p.tm_k;
#pragma unroll
          for (int sub = 0; sub < 2; ++sub)
            tma_load_4d_hint(dst + sub * kBlockBytes, tm, &bar_full[stage], sub * 64, x.hk, 0, phys, policy);
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ================================================================ S^T issuer
    const uint32_t idesc_s = make_idesc_bf16(128, N, false);  // S^T = K . Q^T
    uint32_t kv_it = 0, t = 0;  // ring position and key tiles of this CTA so far
    for (int r = 0;; ++r) {
      KrUnit x;
      if (!take_unit(r, x)) break;
      const int qb = r & 1;
      if (lane == 0) {
        mbar_wait(&bar_q_full[qb], (r >> 1) & 1, abort, p.status, kSiteKrQ);
        const uint64_t dq = make_sdesc_sw128(smem_u32(sQ + qb * C::kQBytes), 16, 1024);
        // S^T of key tile j into S buffer (t + j) & 1, once the softmax has read that buffer's
        // previous scores
        for (int j = 0; j < x.ntiles; ++j) {
          const uint32_t tt = t + j, sb = tt & 1;
          const uint32_t ki = kv_it + 2 * j;
          const int ks = ki % NS;
          mbar_wait(&bar_full[ks], (ki / NS) & 1, abort, p.status, kSiteKrFull);
          if (tt >= 2) mbar_wait(&bar_s_free[sb], ((tt >> 1) - 1) & 1, abort, p.status, kSiteKrSFree);
          tc_fence_after();
          const uint64_t dk = make_sdesc_sw128(smem_u32(sKV + ks * kStageBytes), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kHd / 16; ++kk)
            mma_ss(tmem + sb * N, dk + kmajor_step(kk, kBlockBytes), dq + kmajor_step(kk, C::kRowBytes), idesc_s,
                   kk > 0 ? 1u : 0u);
          mma_commit(&bar_s_full[sb]);
          mma_commit(&bar_empty[ks]);
        }
        mma_commit(&bar_q_empty[qb]);  // the unit's last read of Q (at once when it has no keys)
      }
      __syncwarp();
      t += x.ntiles;
      kv_it += 2 * x.ntiles;
    }
    // drain: every MMA issued has completed before TMEM is released
    if (lane == 0) {
      mma_commit(&bar_drain[0]);
      int no_abort = 0;
      mbar_wait(&bar_drain[0], 0, &no_abort, p.status, kSiteKrDrain);
    }
    __syncwarp();
  } else if (warp == 4) {
    // ================================================================ P V issuer
    const uint32_t idesc_o = make_idesc_bf16_amn(128, N);  // O^T += V^T . P^T (V read MN-major)
    uint32_t kv_it = 0, t = 0;
    for (int r = 0;; ++r) {
      KrUnit x;
      if (!take_unit(r, x)) break;
      const int ob = r & 1;
      const uint32_t tO = tmem + 2 * N + ob * N;
      for (int j = 0; j < x.ntiles; ++j) {
        const uint32_t tt = t + j, sb = tt & 1;
        const uint32_t vi = kv_it + 2 * j + 1;
        const int vs = vi % NS;
        if (lane == 0) mbar_wait(&bar_full[vs], (vi / NS) & 1, abort, p.status, kSiteKrFull);
        __syncwarp();
        {
          // Rows of the sequence's partial last page past kv_len hold no valid value (possibly
          // not even a finite one); P is 0 there but 0 * NaN is NaN, so they are zeroed first.
          const int k0 = (x.kv_t0 + j) * kKeys;
          if (k0 < x.kv_len && x.kv_len < k0 + kKeys && (x.kv_len % p.page_size) != 0) {
            const int r_begin = x.kv_len - k0;
            const int r_end = min(kKeys, ((x.kv_len + p.page_size - 1) / p.page_size) * p.page_size - k0);
            uint8_t* vt = sKV + vs * kStageBytes;
            const int n_chunks = (r_end - r_begin) * 16;  // two 64-column blocks of 8 x 16 bytes per row
            for (int c = lane; c < n_chunks; c += 32) {
              const int row = r_begin + (c >> 4), sub = (c >> 3) & 1;
              *reinterpret_cast<uint4*>(vt + sub * kBlockBytes + row * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
          mbar_wait(&bar_p_full[sb], (tt >> 1) & 1, abort, p.status, kSiteKrP);
          // the unit's first P V overwrites O^T: the epilogue of the unit before last must have read it
          if (j == 0 && r >= 2) mbar_wait(&bar_o_free[ob], ((r >> 1) - 1) & 1, abort, p.status, kSiteKrOFree);
          tc_fence_after();
          const uint64_t dv = make_sdesc_sw128(smem_u32(sKV + vs * kStageBytes), kBlockBytes, 1024);
          const uint64_t dp = make_sdesc_sw128(smem_u32(sP + sb * C::kPBytes), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)
            mma_ss(tO, dv + (uint64_t)kk * (2048 >> 4), dp + kmajor_step(kk, C::kRowBytes), idesc_o,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar_p_free[sb]);
          mma_commit(&bar_empty[vs]);
        }
        __syncwarp();
      }
      if (lane == 0) {
        if (x.ntiles == 0 && r >= 2) mbar_wait(&bar_o_free[ob], ((r >> 1) - 1) & 1, abort, p.status, kSiteKrOFree);
        mma_commit(&bar_o_full[ob]);
      }
      __syncwarp();
      t += x.ntiles;
      kv_it += 2 * x.ntiles;
    }
    if (lane == 0) {
      mma_commit(&bar_drain[1]);
      int no_abort = 0;
      mbar_wait(&bar_drain[1], 0, &no_abort, p.status, kSiteKrDrain);
    }
    __syncwarp();
  } else if (warp >= 5) {
    // ================================================================ softmax
    const int w = warp & 3;                            // TMEM lane quarter
    const int i = w * 32 + lane;                       // key row of a tile; O^T row d in the epilogue
    const uint32_t lane_off = (uint32_t)(w * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t t = 0, xc = 0;  // key tiles and shared-memory exchanges so far
    for (int r = 0;; ++r) {
      KrUnit x;
      if (!take_unit(r, x)) break;
      const int rows = x.q_len * G;  // live columns: column c is token c / G, head hk G + c % G
      const int ob = r & 1;
      const int off = x.kv_len - x.q_len;  // bottom-right causal alignment
      float m[R], l[R];
#pragma unroll
      for (int c = 0; c < R; ++c) {
        m[c] = -INFINITY;
        l[c] = 0.f;
      }
      for (int j = 0; j < x.ntiles; ++j, ++t) {
        const uint32_t sb = t & 1;
        mbar_wait(&bar_s_full[sb], (t >> 1) & 1, abort, p.status, kSiteKrS);
        __syncwarp();
        tc_fence_after();
        uint32_t sr[R];
        tmem_ld_cols<R>(tmem + sb * N + lane_off, sr);
        tc_fence_before();
        mbar_arrive(&bar_s_free[sb]);
        // This thread's key counts for the columns in [lo, hi): none past the keys; under causal
        // masking not the tokens t with key >= off + t + 1, i.e. not the columns c < G (key - off);
        // never the columns past the unit's rows.
        const int key = (x.kv_t0 + j) * kKeys + i;
        int lo = 0, hi = rows;
        if (key >= x.kv_len) {
          hi = 0;
        } else if (p.causal) {
          const int kt = key - off;
          lo = kt <= 0 ? 0 : (kt >= R ? R : min(R, kt * G));
        }
        // Does any of this thread's scores exceed the running maximum by more than the threshold?
        // The four warps' answers are exchanged; only then are the exact column maxima gathered.
        float* xr = &xred[xc & 1][0][0];
        uint64_t* bx = bar_x;
        bool up = false;
#pragma unroll
        for (int c = 0; c < R; ++c) {
          const float s = (c >= lo && c < hi) ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
          sr[c] = __float_as_uint(s);
          up |= s > m[c] + kKrRescaleThreshold;
        }
        up = __any_sync(0xffffffffu, up);
        if (lane == 0) xr[w] = up ? 1.f : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bx[xc & 1]);
        mbar_wait(&bx[xc & 1], (xc >> 1) & 1, abort, p.status, kSiteKrX);
        const float4 votes = *reinterpret_cast<const float4*>(xr);
        ++xc;
        if ((votes.x + votes.y) + (votes.z + votes.w) > 0.f) {
          // rare (the first tile of a unit, or a score far above the running maximum; the same
          // in every thread): the tile's column maxima (a warp reduction, then the four warps'),
          // m raised where they pass the threshold, the partial sums rescaled and, once the
          // previous tile's P V is done, the columns of O^T
          float* xm = &xred[xc & 1][0][0];
#pragma unroll
          for (int c = 0; c < R; ++c) {
            const float tmax = warp_max_f32(__uint_as_float(sr[c]));
            if (lane == 0) xm[c * 4 + w] = tmax;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bx[xc & 1]);
          mbar_wait(&bx[xc & 1], (xc >> 1) & 1, abort, p.status, kSiteKrX);
          ++xc;
          float alpha[R];
#pragma unroll
          for (int c = 0; c < R; ++c) {
            const float4 v = *reinterpret_cast<const float4*>(xm + c * 4);
            const float mt = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
            const bool raise = mt > m[c] + kKrRescaleThreshold;
            alpha[c] = raise ? ex2(m[c] - mt) : 1.f;  // 0 while m is -inf
            m[c] = raise ? mt : m[c];
            l[c] *= alpha[c];
          }
          if (j > 0) {
            const uint32_t tp = t - 1;
            mbar_wait(&bar_p_free[tp & 1], (tp >> 1) & 1, abort, p.status, kSiteKrPFree);
            __syncwarp();
            tc_fence_after();
            const uint32_t tO = tmem + 2 * N + ob * N + lane_off;
            uint32_t o[R];
            tmem_ld_cols<R>(tO, o);
#pragma unroll
            for (int c = 0; c < R; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha[c]);
            tmem_st_cols<R>(tO, o);
            tmem_st_wait();
          }
        }
        // P^T (bf16) into its swizzled K-major buffer: row c, key i (0 where masked)
        if (t >= 2) mbar_wait(&bar_p_free[sb], ((t >> 1) - 1) & 1, abort, p.status, kSiteKrPFree);
        uint8_t* prow = sP + sb * C::kPBytes + (i >> 6) * C::kRowBytes + (i & 7) * 2;
        const int ch = (i & 63) >> 3;
#pragma unroll
        for (int c = 0; c < R; ++c) {
          const float e = ex2(__uint_as_float(sr[c]) - (m[c] == -INFINITY ? 0.f : m[c]));
          l[c] += e;
          const int row = c;
          *reinterpret_cast<__nv_bfloat16*>(prow + row * 128 + ((ch ^ (row & 7)) << 4)) = __float2bfloat16_rn(e);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar_p_full[sb]);
      }
      // ------------------------------------------------------------ epilogue
      // l per column over the 128 key rows: a warp sum, then the four warps' sums
      float* xr = &xred[xc & 1][0][0];
      uint64_t* bx = bar_x;
#pragma unroll
      for (int c = 0; c < R; ++c) {
        float v = l[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) xr[c * 4 + w] = v;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bx[xc & 1]);
      mbar_wait(&bx[xc & 1], (xc >> 1) & 1, abort, p.status, kSiteKrX);
      ++xc;
#pragma unroll
      for (int c = 0; c < R; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(xr + c * 4);
        l[c] = (v.x + v.y) + (v.z + v.w);
      }
      mbar_wait(&bar_o_full[ob], (r >> 1) & 1, abort, p.status, kSiteKrO);
      __syncwarp();
      tc_fence_after();
      uint32_t orr[R];
      if (x.ntiles > 0) {
        tmem_ld_cols<R>(tmem + 2 * N + ob * N + lane_off, orr);
      } else {
#pragma unroll
        for (int c = 0; c < R; ++c) orr[c] = 0u;
      }
      tc_fence_before();
      mbar_arrive(&bar_o_free[ob]);  // the MMA may now overwrite this O^T buffer (unit r + 2)
      // O[token][head][d = i] = O^T[i][c] / l_c; a split unit writes its fp32 partial state
      float* o_f32 = p.o_f32;
      float* lse_out = p.lse;
      int64_t row_base = 0;
      if (p.kv_splits > 1) {
        o_f32 = p.o_part;
        lse_out = p.lse_part;
        row_base = (int64_t)x.split * p.total_q * p.Hq;
      }
      int tq = 0, g = 0;  // token and head of column c
#pragma unroll
      for (int c = 0; c < R; ++c) {
        const int64_t tok = x.tok0 + tq;
        if (c < rows && tok < p.total_q) {
          const int64_t orow = row_base + tok * p.Hq + x.hk * G + g;
          const float inv = l[c] > 0.f ? 1.f / l[c] : 0.f;
          const float o = __uint_as_float(orr[c]) * inv;
          if (o_f32 != nullptr) {
            o_f32[orow * kHd + i] = o;
          } else {
            reinterpret_cast<__nv_bfloat16*>(p.o)[orow * kHd + i] = __float2bfloat16_rn(o);
          }
          if (i == c && lse_out != nullptr)
            lse_out[orow] = l[c] > 0.f ? (m[c] + __log2f(l[c])) * kKrLn2 : -INFINITY;
        }
        if (++g == G) {
          g = 0;
          ++tq;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int R>
cudaError_t launch_decode_tc_impl(const PrefillParams& p, int grid, cudaStream_t stream, bool programmatic) {
  constexpr int N = 16;
  auto kern = decode_tc_kernel<N, R>;
  static std::atomic<unsigned> configured_mask{0u};  // one bit per device ordinal below 32
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 32 || !(configured_mask.load(std::memory_order_acquire) & (1u << dev))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, KrCfg<N>::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 32) configured_mask.fetch_or(1u << dev, std::memory_order_release);
  }
  // programmatic stream serialization: the CTAs may start (barrier set-up, TMEM allocation) while
  // the planning kernel before them runs; they wait for it before reading its results
  if (!programmatic) {
    kern<<<grid, 288, KrCfg<N>::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(288);
  cfg.dynamicSmemBytes = KrCfg<N>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

int decode_tc_columns(int max_q_len, int group, int d, int max_rows) {
  if (d != kHd || max_q_len < 1 || group < 1) return 0;
  const long long rows = (long long)max_q_len * group;
  if (rows > max_rows || rows > 16) return 0;
  int r = 4;
  while (r < rows) r *= 2;
  return r;
}

cudaError_t launch_decode_tc(const PrefillParams& p, int columns, int sm_count, int max_items, int max_kv_tiles,
                             int2* work_list, int* work_count, cudaStream_t stream, cudaEvent_t after_plan) {
  cudaError_t e = launch_plan_paged(p, max_items, max_kv_tiles, work_list, work_count, stream);
  if (e == cudaSuccess && after_plan != nullptr) e = cudaEventRecord(after_plan, stream);
  if (e != cudaSuccess) return e;
  const long long units = (long long)max_items * p.Hkv * p.kv_splits;  // an upper bound
  const int grid = (int)(units < sm_count ? units : sm_count);
  if (grid <= 0) return cudaSuccess;
  switch (columns) {
    // with an event recorded between the plan and this kernel, an ordinary launch
    case 4: return launch_decode_tc_impl<4>(p, grid, stream, after_plan == nullptr);
    case 8: return launch_decode_tc_impl<8>(p, grid, stream, after_plan == nullptr);
    case 16: return launch_decode_tc_impl<16>(p, grid, stream, after_plan == nullptr);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
