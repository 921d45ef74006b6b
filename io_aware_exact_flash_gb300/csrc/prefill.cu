// Tensor-core attention forward for sm_103a: the tiled, fused method of "I/O-Aware Kernels"
// (datasystem.school, Module 5), section "FlashAttention: tiling + online softmax". A query tile
// stays in shared memory, key/value tiles stream through a TMA-fed ring, S = Q K^T and O += P V run
// as tcgen05 MMAs with their accumulators in tensor memory (TMEM), and the softmax is computed
// online (running max m, running sum l, rescaled O), so no score ever reaches device memory.
//
// One kernel serves the dense layout and the paged/ragged layout of the page's section
// "FlashInfer: I/O-aware attention for serving"; they differ only in how tiles are addressed.
//
// CTA organisation (384 threads, one CTA per SM):
//   warp 0      TMA producer: Q tiles once, then K_0, V_0, K_1, V_1, ... into a ring of stages
//   warp 1      TMEM owner and MMA issuer (one elected lane issues every tcgen05.mma)
//   warps 2-3   idle
//   warps 4-7   softmax warpgroup 0 -> query tile 0 (rows 0..127 of the CTA's 256)
//   warps 8-11  softmax warpgroup 1 -> query tile 1 (rows 128..255)
// The two warpgroups ping-pong: while one computes its softmax the tensor core runs the other's
// P V and next Q K^T.
//
// TMEM columns: S/P of tile g at [128 g, 128 g + 128) (P, as packed bf16 pairs, overwrites the
// first 64 columns of S), O of tile g at [256 + g D, 256 + (g+1) D).
#include <cuda_bf16.h>
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
  static constexpr int kStages = D == 128 ? 4 : 8;
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
};

template <int D, bool PAGED>
__global__ void __launch_bounds__(kPrefillThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = Cfg<D>;
  constexpr int NS = C::kStages;
  constexpr int TB = C::kTileBytes;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                  // kQTiles tiles
  uint8_t* sKV = smem + kQTiles * TB;  // NS stages

  __shared__ uint64_t bar_q[kQTiles], bar_full[NS], bar_empty[NS];
  __shared__ uint64_t bar_s[kQTiles], bar_p[kQTiles], bar_o[kQTiles], bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ------------------------------------------------------------------ work unit
  int seq, h, qt2, q_len, kv_len;
  int64_t tok0;  // token index of the sequence's first query row
  if constexpr (PAGED) {
    const int item = blockIdx.x / p.Hq;
    h = blockIdx.x % p.Hq;
    if (item >= *p.work_count) return;  // grid is an upper bound on the number of items
    const int2 w = p.work_list[item];
    seq = w.x;
    qt2 = w.y;
    const int c0 = p.cu_seqlens_q[seq], c1 = p.cu_seqlens_q[seq + 1];
    tok0 = c0;
    q_len = c1 - c0;
    kv_len = p.kv_lens[seq];
  } else {
    const int bh_count = p.B * p.Hq;
    const int n2 = (p.S + 2 * kBM - 1) / (2 * kBM);
    const int x = blockIdx.x;
    // causal work is heaviest for the last query tiles: launch those first
    qt2 = p.causal ? (n2 - 1 - x / bh_count) : (x / bh_count);
    const int bh = x % bh_count;
    seq = bh / p.Hq;
    h = bh % p.Hq;
    tok0 = (int64_t)seq * p.S;
    q_len = p.S;
    kv_len = p.S;
  }
  const int hk = h / p.group;
  const int off = kv_len - q_len;  // bottom-right causal alignment
  int nkv[kQTiles], row0[kQTiles];
  int nmax = 0;
#pragma unroll
  for (int g = 0; g < kQTiles; ++g) {
    row0[g] = qt2 * (2 * kBM) + g * kBM;
    if (row0[g] >= q_len) {
      nkv[g] = -1;  // no query rows in this tile
    } else {
      const int last = min(row0[g] + kBM - 1, q_len - 1);
      const int lim = p.causal ? min(kv_len, last + off + 1) : kv_len;
      nkv[g] = lim > 0 ? (lim + kBN - 1) / kBN : 0;
    }
    nmax = max(nmax, nkv[g]);
  }

  // ------------------------------------------------------------------ setup
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int g = 0; g < kQTiles; ++g) {
      mbar_init(&bar_q[g], 1);
      mbar_init(&bar_s[g], 1);
      mbar_init(&bar_p[g], 4 * 32);
      mbar_init(&bar_o[g], 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_drain, 1);
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

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      for (int g = 0; g < kQTiles; ++g) {
        if (nkv[g] <= 0) continue;
        mbar_arrive_expect_tx(&bar_q[g], TB);
        const int qrow = PAGED ? (int)(tok0 + row0[g]) : row0[g];
        const int qbat = PAGED ? 0 : seq;
#pragma unroll
        for (int sub = 0; sub < C::kSub; ++sub)
          tma_load_4d(sQ + g * TB + sub * C::kSubBytes, &p.tm_q, &bar_q[g], sub * 64, h, qrow, qbat);
      }
    }
    const uint64_t kv_policy = policy_evict_last();
    for (int idx = 0; idx < 2 * nmax; ++idx) {
      const int j = idx >> 1;
      const bool is_v = idx & 1;
      const int stage = idx % NS;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&bar_empty[stage], ((idx / NS) & 1) ^ 1, abort, p.status, kSiteProducerEmpty);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      uint8_t* dst = sKV + stage * TB;
      const CUtensorMap* tm = is_v ? &p.tm_v : &p.tm_k;
      if (lane == 0) mbar_arrive_expect_tx(&bar_full[stage], TB);
      __syncwarp();
      if constexpr (!PAGED) {
        if (lane == 0) {
#pragma unroll
          for (int sub = 0; sub < C::kSub; ++sub)
            tma_load_4d_hint(dst + sub * C::kSubBytes, tm, &bar_full[stage], sub * 64, hk, j * kBN, seq, kv_policy);
        }
      } else {
        const int ppt = kBN / p.page_size;  // pages per tile
        if (lane < ppt) {
          const int lp = j * ppt + lane;    // logical page of this sequence
          int phys = p.num_pages;           // past the pool: TMA fills zeros
          if (lp * p.page_size < kv_len && lp < p.max_pages_per_seq)
            phys = p.page_table[(int64_t)seq * p.max_pages_per_seq + lp];
#pragma unroll
          for (int sub = 0; sub < C::kSub; ++sub)
            tma_load_4d_hint(dst + sub * C::kSubBytes + lane * p.page_size * 128, tm, &bar_full[stage], sub * 64,
                             hk, 0, phys, kv_policy);
        }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    const uint32_t idesc_s = make_idesc_bf16(kBM, kBN, false);
    const uint32_t idesc_pv = make_idesc_bf16(kBM, D, true);
    const uint32_t sQa = smem_u32(sQ), sKVa = smem_u32(sKV);
    // K-major operands (Q, K): 16-element K steps advance 32 bytes inside a 128-byte swizzle row,
    // and every 4 steps move to the next 16 KB column block.
    auto kmaj = [&](uint32_t base, int kk) {
      return make_sdesc_sw128(base + (kk >> 2) * C::kSubBytes + (kk & 3) * 32, 16, 1024);
    };
    // V as the MN-major B operand of P V: 16 keys = 16 rows of 128 bytes per K step; the two
    // 64-column blocks of d sit 16 KB apart (leading-dimension offset).
    auto vmaj = [&](uint32_t base, int kk) { return make_sdesc_sw128(base + kk * 2048, C::kSubBytes, 1024); };

    if (lane == 0) {
      for (int g = 0; g < kQTiles; ++g)
        if (nkv[g] > 0) mbar_wait(&bar_q[g], 0, abort, p.status, kSiteMmaQ);
    }
    if (nmax > 0) {
      if (lane == 0) {
        mbar_wait(&bar_full[0], 0, abort, p.status, kSiteMmaFull);
        tc_fence_after();
        for (int g = 0; g < kQTiles; ++g) {
          if (nkv[g] <= 0) continue;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + g * 128, kmaj(sQa + g * TB, kk), kmaj(sKVa, kk), idesc_s, kk > 0);
          mma_commit(&bar_s[g]);
        }
        mma_commit(&bar_empty[0]);
      }
      for (int j = 0; j < nmax; ++j) {
        const int vi = 2 * j + 1, ki = 2 * j + 2;
        const int vs = vi % NS, ks = ki % NS;
        const bool has_next = j + 1 < nmax;
        if (lane == 0) {
          mbar_wait(&bar_full[vs], (vi / NS) & 1, abort, p.status, kSiteMmaFull);
          if (has_next) mbar_wait(&bar_full[ks], (ki / NS) & 1, abort, p.status, kSiteMmaFull);
        }
        __syncwarp();
        if constexpr (PAGED) {
          // Rows of the sequence's partial last page past kv_len hold no valid value (possibly
          // not even a finite one); P is 0 there but 0 * NaN is NaN, so they are zeroed first.
          const int t0 = j * kBN;
          if (t0 < kv_len && kv_len < t0 + kBN && (kv_len % p.page_size) != 0) {
            const int r_begin = kv_len - t0;
            const int r_end = min(kBN, ((kv_len + p.page_size - 1) / p.page_size) * p.page_size - t0);
            uint8_t* vt = sKV + vs * TB;
            const int n_chunks = (r_end - r_begin) * C::kSub * 8;  // 16-byte chunks
            for (int c = lane; c < n_chunks; c += 32) {
              const int row = r_begin + c / (C::kSub * 8);
              const int sub = (c / 8) % C::kSub;
              *reinterpret_cast<uint4*>(vt + sub * C::kSubBytes + row * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          for (int g = 0; g < kQTiles; ++g) {
            if (j >= nkv[g]) continue;
            mbar_wait(&bar_p[g], j & 1, abort, p.status, kSiteMmaP);
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              mma_ts(tmem + C::kColO + g * D, tmem + g * 128 + kk * 8, vmaj(sKVa + vs * TB, kk), idesc_pv,
                     (j > 0 || kk > 0) ? 1u : 0u);
            if (j == nkv[g] - 1) mma_commit(&bar_o[g]);
            if (j + 1 < nkv[g]) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tmem + g * 128, kmaj(sQa + g * TB, kk), kmaj(sKVa + ks * TB, kk), idesc_s, kk > 0);
              mma_commit(&bar_s[g]);
            }
          }
          mma_commit(&bar_empty[vs]);
          if (has_next) mma_commit(&bar_empty[ks]);
        }
        __syncwarp();
      }
    }
    // drain: every MMA this CTA issued has completed before TMEM is released
    if (lane == 0) {
      mma_commit(&bar_drain);
      int no_abort = 0;
      mbar_wait(&bar_drain, 0, &no_abort, p.status, kSiteDrain);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ================================================================ softmax warpgroups
    const int g = (warp - 4) >> 2;
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + g * 128 + lane_off;
    const uint32_t tO = tmem + C::kColO + g * D + lane_off;
    if (nkv[g] >= 0) {
      const int row = row0[g] + r;
      const int lim_row = p.causal ? min(kv_len, row + off + 1) : kv_len;  // keys [0, lim_row)
      const float sl2 = p.scale_log2;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkv[g]; ++j) {
        mbar_wait(&bar_s[g], j & 1, abort, p.status, kSiteSoftmaxS);
        __syncwarp();  // lanes leave the wait at different times; tcgen05.ld is warp-collective
        tc_fence_after();
        uint32_t sr[kBN];
        tmem_ld32(tS + 0, sr + 0);
        tmem_ld32(tS + 32, sr + 32);
        tmem_ld32(tS + 64, sr + 64);
        tmem_ld32(tS + 96, sr + 96);
        tmem_ld_wait(sr + 0);
        tmem_ld_wait(sr + 32);
        tmem_ld_wait(sr + 64);
        tmem_ld_wait(sr + 96);
        const int valid = lim_row - j * kBN;
        if (valid < kBN) {
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c >= valid) sr[c] = 0xff800000u;  // -inf
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBN; ++c) mx = fmaxf(mx, u2f(sr[c]));
        const float m_tile = mx * sl2;
        float alpha = 1.f;
        const bool need = m_tile > m_run + kRescaleThreshold;
        if (need) {
          alpha = ex2(m_run - m_tile);  // 0 while m_run is -inf
          m_run = m_tile;
        }
        l_run *= alpha;
        const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p0 = ex2(fmaf(u2f(sr[cc * 32 + 2 * i]), sl2, neg_m));
            const float p1 = ex2(fmaf(u2f(sr[cc * 32 + 2 * i + 1]), sl2, neg_m));
            l_run += p0 + p1;
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + cc * 16, pk);
        }
        // O rescale (after P is written, so S no longer occupies registers): P V of the previous
        // tile is complete, because the commit that signalled this tile's S was issued after it.
        if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32(tO + cc * 32, orr);
            tmem_ld_wait(orr);
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = f2u(u2f(orr[i]) * alpha);
            tmem_st32(tO + cc * 32, orr);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_p[g]);
        __syncwarp();
      }
      // ---------------------------------------------------------- epilogue: O / l, LSE
      if (nkv[g] > 0) {
        mbar_wait(&bar_o[g], 0, abort, p.status, kSiteSoftmaxO);
        __syncwarp();
        tc_fence_after();
      }
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const int64_t tok = tok0 + row;
      const bool store = row < q_len && (!PAGED || tok < p.total_q);
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + (tok * p.Hq + h) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t orr[32];
        if (nkv[g] > 0) {
          tmem_ld32(tO + cc * 32, orr);
          tmem_ld_wait(orr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(u2f(orr[2 * i]) * inv_l, u2f(orr[2 * i + 1]) * inv_l);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (store && p.lse != nullptr)
        p.lse[tok * p.Hq + h] = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Work list for the paged prefill: one item per (sequence, pair of query tiles), sorted by the
// number of key tiles it streams, heaviest first (a counting sort over that cost).
__global__ void plan_paged_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ kv_lens,
                                  int num_seqs, int causal, int max_cost, int max_items,
                                  int2* __restrict__ work_list, int* __restrict__ work_count) {
  extern __shared__ int hist[];  // max_cost + 1 buckets
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int c = tid; c <= max_cost; c += nt) hist[c] = 0;
  __syncthreads();
  auto cost_of = [&](int q_len, int kv_len, int it) {
    const int last = min(it * 2 * kBM + 2 * kBM - 1, q_len - 1);
    const int lim = causal ? min(kv_len, last + (kv_len - q_len) + 1) : kv_len;
    const int n = lim > 0 ? (lim + kBN - 1) / kBN : 0;
    return min(n, max_cost);
  };
  for (int s = tid; s < num_seqs; s += nt) {
    const int q_len = cu[s + 1] - cu[s], kv_len = kv_lens[s];
    const int items = (q_len + 2 * kBM - 1) / (2 * kBM);
    for (int it = 0; it < items; ++it) atomicAdd(&hist[cost_of(q_len, kv_len, it)], 1);
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int c = max_cost; c >= 0; --c) {
      const int t = hist[c];
      hist[c] = run;
      run += t;
    }
    *work_count = min(run, max_items);  // more items than the host bound means inconsistent lengths
  }
  __syncthreads();
  for (int s = tid; s < num_seqs; s += nt) {
    const int q_len = cu[s + 1] - cu[s], kv_len = kv_lens[s];
    const int items = (q_len + 2 * kBM - 1) / (2 * kBM);
    for (int it = 0; it < items; ++it) {
      const int pos = atomicAdd(&hist[cost_of(q_len, kv_len, it)], 1);
      if (pos < max_items) work_list[pos] = make_int2(s, it);
    }
  }
}

template <int D, bool PAGED>
cudaError_t launch_prefill_impl(const PrefillParams& p, int grid, cudaStream_t stream) {
  auto kern = prefill_kernel<D, PAGED>;
  static int configured_mask = 0;  // one bit per device ordinal below 32
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 32 || !(configured_mask & (1 << dev))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 32) configured_mask |= (1 << dev);
  }
  kern<<<grid, kPrefillThreads, Cfg<D>::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_dense(const PrefillParams& p, int d, cudaStream_t stream) {
  const int n2 = (p.S + 2 * kBM - 1) / (2 * kBM);
  const int grid = n2 * p.B * p.Hq;
  if (d == 128) return launch_prefill_impl<128, false>(p, grid, stream);
  return launch_prefill_impl<64, false>(p, grid, stream);
}

cudaError_t launch_prefill_paged(const PrefillParams& p, int d, int max_items, int max_kv_tiles, int2* work_list,
                                 int* work_count, cudaStream_t stream) {
  const int smem = (max_kv_tiles + 1) * (int)sizeof(int);
  plan_paged_kernel<<<1, 1024, smem, stream>>>(p.cu_seqlens_q, p.kv_lens, p.num_seqs, p.causal, max_kv_tiles,
                                              max_items, work_list, work_count);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int grid = max_items * p.Hq;
  if (d == 128) return launch_prefill_impl<128, true>(p, grid, stream);
  return launch_prefill_impl<64, true>(p, grid, stream);
}

}  // namespace fa
