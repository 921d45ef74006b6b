// Split-KV decode over a paged KV cache, and the LSE-weighted merge of partial attention states.
//
// Decoding attends one query token per sequence to that sequence's whole key set, read through
// its page table ("I/O-Aware Kernels", datasystem.school Module 5, section "FlashInfer: I/O-aware
// attention for serving"). Every key/value byte is used by the Hq/Hkv query heads of one group
// and by nothing else, so the work is a stream over the cache at a few flops per byte: it is
// bound by HBM bandwidth, not by math. This kernel runs it on the CUDA cores, reading each K/V
// byte exactly once with enough bytes in flight to keep HBM busy. fa_paged_fwd sends decode
// batches to the tensor-core kernel instead (prefill.cu: GQA packing and key splits), which
// measured faster for every group; this kernel serves fa_paged_decode_noalloc and, with the
// environment variable FA_DECODE_TC=0, fa_paged_fwd's decode batches of groups 1, 2, 4 and 8.
//
// Grid: (split, sequence, kv-head block). A CTA streams 16-row blocks of its sequence's pages
// (one page when page_size = 16) through a ring of shared-memory stages filled by bulk async
// copies, one warp per kv head; lane 0 of warp 0 refills a stage as soon as all warps release
// it. Each warp keeps its group's query heads in registers, computes the scores of 16 rows,
// updates the running max m and sum l once per block, and accumulates O += p v. A CTA writes
// one partial state per (split, query head): O normalised over its keys and its LSE; the last
// CTA of a sequence to finish merges the splits (with one split the CTA writes the final O and
// LSE itself).
#include <cuda_bf16.h>
#include <atomic>
#include "kernels.cuh"

namespace fa {

namespace {

constexpr int kRowsPerBlock = 16;  // rows per ring stage
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxHeadsPerCta = 8;

enum : uint32_t { kSiteDecodeEmpty = 16, kSiteDecodeFull = 17, kSiteDecodeBadPage = 18 };

template <int D, int G>
struct DecodeCfg {
  // lanes cooperating on one key row: enough that each lane holds <= 64 accumulators
  static constexpr int LPR = (G * D / 8 <= 64) ? 8 : 16;
  static constexpr int EPL = D / LPR;      // elements per lane (multiple of 8)
  static constexpr int CPL = EPL / 8;      // 16-byte chunks per lane
  static constexpr int RPI = 32 / LPR;     // rows a warp handles per step
  static constexpr int ITERS = kRowsPerBlock / RPI;
  // a block is taken in SUB sub-blocks of SITERS steps (one max / rescale each), so that the
  // scores held at once (SITERS x G per lane) stay within 16 registers where they would exceed 32
  static constexpr int SUB = (ITERS * G > 32) ? 4 : 1;
  static constexpr int SITERS = ITERS / SUB;
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// bf16 x 8 -> four fp32 pairs (element 2i in the low half of pair i)
__device__ __forceinline__ void bf16x8_to_f32x2(const uint4 u, uint64_t* f2) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) f2[i] = f32x2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

template <int D, int G>
__global__ void __launch_bounds__(kMaxHeadsPerCta * 32, 1)
    decode_kernel(const __grid_constant__ DecodeParams p, int n_stages) {
  using C = DecodeCfg<D, G>;
  const int split = blockIdx.x, seq = blockIdx.y;
  const int hpc = p.heads_per_cta;
  const int hk0 = blockIdx.z * hpc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int q_begin = p.cu_seqlens_q[seq];
  const int q_len = p.cu_seqlens_q[seq + 1] - q_begin;
  if (q_len <= 0 || q_begin < 0 || q_begin >= p.total_q) return;  // no query row of this sequence
  const int kv_len = min(p.kv_lens[seq], p.max_pages_per_seq * p.page_size);
  const int n_blocks = (kv_len + kRowsPerBlock - 1) / kRowsPerBlock;
  const int blk_begin = split * p.pages_per_split * (p.page_size / kRowsPerBlock);
  const int blk_end = min(n_blocks, blk_begin + p.pages_per_split * (p.page_size / kRowsPerBlock));
  const int n_mine = max(0, blk_end - blk_begin);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int chunk = kRowsPerBlock * hpc * D * 2;  // bytes of K (or V) per stage
  __shared__ uint64_t bar_full[8], bar_empty[8];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < n_stages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], hpc);
    }
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;

  // Producer role (lane 0 of warp 0): fill stage s with block i, both K and V.
  const uint64_t pol = policy_evict_first();
  const int blocks_per_page = p.page_size / kRowsPerBlock;
  const int64_t row_bytes = (int64_t)p.Hkv * D * 2;  // one slot of a page, all kv heads
  auto issue = [&](int i) {
    const int s = i % n_stages;
    const int blk = blk_begin + i;
    const int lp = blk / blocks_per_page;
    const int slot0 = (blk % blocks_per_page) * kRowsPerBlock;
    int phys = p.page_table[(int64_t)seq * p.max_pages_per_seq + lp];
    if (phys < 0 || phys >= p.num_pages) {  // never read outside the pool: record and use page 0
      if (p.status) {
        atomicCAS(&p.status->code, 0u, 8u /* FA_ERR_DEVICE_BAD_PAGE */);
        atomicExch(&p.status->where, kSiteDecodeBadPage);
      }
      phys = 0;
    }
    uint8_t* dk = smem + (size_t)s * 2 * chunk;
    uint8_t* dv = dk + chunk;
    mbar_arrive_expect_tx(&bar_full[s], 2 * chunk);
    const int64_t base = ((int64_t)phys * p.page_size + slot0) * row_bytes + (int64_t)hk0 * D * 2;
    const uint8_t* gk = reinterpret_cast<const uint8_t*>(p.k_pages) + base;
    const uint8_t* gv = reinterpret_cast<const uint8_t*>(p.v_pages) + base;
    if (hpc * D * 2 == row_bytes) {  // the block's rows are contiguous for all kv heads
      bulk_load_hint(dk, gk, chunk, &bar_full[s], pol);
      bulk_load_hint(dv, gv, chunk, &bar_full[s], pol);
    } else {
      for (int r = 0; r < kRowsPerBlock; ++r) {
        bulk_load_hint(dk + r * hpc * D * 2, gk + r * row_bytes, hpc * D * 2, &bar_full[s], pol);
        bulk_load_hint(dv + r * hpc * D * 2, gv + r * row_bytes, hpc * D * 2, &bar_full[s], pol);
      }
    }
  };
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < min(n_stages, n_mine); ++i) issue(i);
  }

  // -------------------------------------------------------------- consumers: one warp per kv head
  const int hk = hk0 + warp;
  const int rg = lane / C::LPR;  // row within a step
  const int lr = lane % C::LPR;  // lane within the row
  const int tok = q_begin;       // the single query token of this sequence
  // q and the output accumulator are held as fp32 pairs for the paired .f32x2 instructions
  uint64_t qf2[G][C::EPL / 2];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int h = hk * G + g;
    const uint4* qp = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + ((int64_t)tok * p.Hq + h) * D);
#pragma unroll
    for (int c = 0; c < C::CPL; ++c) {
      float t[8];
      bf16x8_to_f32(qp[lr + c * C::LPR], t);
#pragma unroll
      for (int e = 0; e < 4; ++e) qf2[g][c * 4 + e] = f32x2(t[2 * e] * p.scale_log2, t[2 * e + 1] * p.scale_log2);
    }
  }
  float m[G], l[G];
  uint64_t o2[G][C::EPL / 2];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < C::EPL / 2; ++e) o2[g][e] = 0ull;
  }

  for (int i = 0; i < n_mine; ++i) {
    const int s = i % n_stages;
    mbar_wait(&bar_full[s], (i / n_stages) & 1, abort, p.status, kSiteDecodeFull);
    const uint8_t* sk = smem + (size_t)s * 2 * chunk;
    const uint8_t* sv = sk + chunk;
    const int row_base = (blk_begin + i) * kRowsPerBlock;
#pragma unroll
    for (int hb = 0; hb < C::SUB; ++hb) {
      float sc[C::SITERS][G];
#pragma unroll
      for (int it = 0; it < C::SITERS; ++it) {
        const int r = (hb * C::SITERS + it) * C::RPI + rg;
        const uint4* kp = reinterpret_cast<const uint4*>(sk + ((size_t)r * hpc + warp) * D * 2);
        uint64_t kf2[C::EPL / 2];
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) bf16x8_to_f32x2(kp[lr + c * C::LPR], &kf2[c * 4]);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          uint64_t acc2 = 0ull;
#pragma unroll
          for (int e = 0; e < C::EPL / 2; ++e) acc2 = fma_f32x2(qf2[g][e], kf2[e], acc2);
          float a0, a1;
          split_f32x2(acc2, a0, a1);
          float acc = a0 + a1;
#pragma unroll
          for (int sh = 1; sh < C::LPR; sh <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
          sc[it][g] = (row_base + r < kv_len) ? acc : -INFINITY;
        }
      }
      // one max / rescale per sub-block
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float bm = sc[0][g];
#pragma unroll
        for (int it = 1; it < C::SITERS; ++it) bm = fmaxf(bm, sc[it][g]);
#pragma unroll
        for (int sh = C::LPR; sh < 32; sh <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, sh));
        const float m_new = fmaxf(m[g], bm);
        if (m_new > m[g]) {
          const float alpha = ex2(m[g] - m_new);  // 0 while m is -inf
          l[g] *= alpha;
          const uint64_t a2 = f32x2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < C::EPL / 2; ++e) o2[g][e] = mul_f32x2(o2[g][e], a2);
          m[g] = m_new;
        }
        const float mu = (m[g] == -INFINITY) ? 0.f : m[g];
#pragma unroll
        for (int it = 0; it < C::SITERS; ++it) {
          sc[it][g] = ex2(sc[it][g] - mu);
          l[g] += sc[it][g];
        }
      }
#pragma unroll
      for (int it = 0; it < C::SITERS; ++it) {
        const int r = (hb * C::SITERS + it) * C::RPI + rg;
        const uint4* vp = reinterpret_cast<const uint4*>(sv + ((size_t)r * hpc + warp) * D * 2);
        uint64_t vf2[C::EPL / 2];
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) bf16x8_to_f32x2(vp[lr + c * C::LPR], &vf2[c * 4]);
        // rows past kv_len carry p = 0; their V may be arbitrary bits, so they are skipped
        if (row_base + r < kv_len) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const uint64_t p2 = f32x2(sc[it][g], sc[it][g]);
#pragma unroll
            for (int e = 0; e < C::EPL / 2; ++e) o2[g][e] = fma_f32x2(p2, vf2[e], o2[g][e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar_empty[s]);
    // refill this stage once every warp has released it
    if (warp == 0 && lane == 0 && i + n_stages < n_mine) {
      if (mbar_wait(&bar_empty[s], (i / n_stages) & 1, abort, p.status, kSiteDecodeEmpty)) issue(i + n_stages);
    }
  }
  float o[G][C::EPL];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < C::EPL / 2; ++e) split_f32x2(o2[g][e], o[g][2 * e], o[g][2 * e + 1]);

  // combine the row groups of the warp (they share m): sum l and O over lanes lr + k * LPR
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int sh = C::LPR; sh < 32; sh <<= 1) {
      l[g] += __shfl_xor_sync(0xffffffffu, l[g], sh);
#pragma unroll
      for (int e = 0; e < C::EPL; ++e) o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], sh);
    }
  }
  if (rg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int h = hk * G + g;
      const float inv_l = l[g] > 0.f ? 1.f / l[g] : 0.f;
      const float lse2 = l[g] > 0.f ? m[g] + __log2f(l[g]) : -INFINITY;
      if (p.num_splits == 1 && p.o_f32 != nullptr) {
        float4* op = reinterpret_cast<float4*>(p.o_f32 + ((int64_t)tok * p.Hq + h) * D);
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) {
          op[2 * (lr + c * C::LPR)] = make_float4(o[g][c * 8 + 0] * inv_l, o[g][c * 8 + 1] * inv_l,
                                                  o[g][c * 8 + 2] * inv_l, o[g][c * 8 + 3] * inv_l);
          op[2 * (lr + c * C::LPR) + 1] = make_float4(o[g][c * 8 + 4] * inv_l, o[g][c * 8 + 5] * inv_l,
                                                      o[g][c * 8 + 6] * inv_l, o[g][c * 8 + 7] * inv_l);
        }
        if (lr == 0 && p.lse) p.lse[(int64_t)tok * p.Hq + h] = lse2 * kLn2;
      } else if (p.num_splits == 1) {
        __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(p.o) + ((int64_t)tok * p.Hq + h) * D;
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) {
          uint4 w;
          w.x = pack_bf16x2(o[g][c * 8 + 0] * inv_l, o[g][c * 8 + 1] * inv_l);
          w.y = pack_bf16x2(o[g][c * 8 + 2] * inv_l, o[g][c * 8 + 3] * inv_l);
          w.z = pack_bf16x2(o[g][c * 8 + 4] * inv_l, o[g][c * 8 + 5] * inv_l);
          w.w = pack_bf16x2(o[g][c * 8 + 6] * inv_l, o[g][c * 8 + 7] * inv_l);
          reinterpret_cast<uint4*>(op)[lr + c * C::LPR] = w;
        }
        if (lr == 0 && p.lse) p.lse[(int64_t)tok * p.Hq + h] = lse2 * kLn2;
      } else {
        const int64_t prow = ((int64_t)split * p.num_seqs + seq) * p.Hq + h;
        if (l[g] > 0.f) {
          float4* op = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
          for (int c = 0; c < C::CPL; ++c) {
            op[2 * (lr + c * C::LPR)] = make_float4(o[g][c * 8 + 0] * inv_l, o[g][c * 8 + 1] * inv_l,
                                                    o[g][c * 8 + 2] * inv_l, o[g][c * 8 + 3] * inv_l);
            op[2 * (lr + c * C::LPR) + 1] = make_float4(o[g][c * 8 + 4] * inv_l, o[g][c * 8 + 5] * inv_l,
                                                        o[g][c * 8 + 6] * inv_l, o[g][c * 8 + 7] * inv_l);
          }
        }
        if (lr == 0) p.lse_part[prow] = lse2;
      }
    }
  }
  if (p.num_splits == 1) return;

  // ---------------------------------------------------------------- LSE-weighted merge
  // The last CTA of this (sequence, kv-head block) to finish merges every split:
  //   lse = log2 sum_s 2^{lse_s},  O = sum_s 2^{lse_s - lse} O_s
  // (log2 domain, scaled scores). A split with lse_s = -inf had no keys; its O_s is not read.
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&p.counters[(int64_t)seq * gridDim.z + blockIdx.z], 1);
    is_last = (prev == p.num_splits - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  constexpr int kPerHead = D / 4;
  for (int t = threadIdx.x; t < hpc * G * kPerHead; t += blockDim.x) {
    const int h = hk0 * G + t / kPerHead, e4 = t % kPerHead;
    float mx = -INFINITY;
    for (int sp = 0; sp < p.num_splits; ++sp)
      mx = fmaxf(mx, __ldcg(&p.lse_part[((int64_t)sp * p.num_seqs + seq) * p.Hq + h]));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (mx != -INFINITY) {
      for (int sp = 0; sp < p.num_splits; ++sp) {
        const int64_t prow = ((int64_t)sp * p.num_seqs + seq) * p.Hq + h;
        const float ls = __ldcg(&p.lse_part[prow]);
        if (ls == -INFINITY) continue;
        const float wgt = ex2(ls - mx);
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.o_part + prow * D) + e4);
        acc.x = fmaf(wgt, v.x, acc.x);
        acc.y = fmaf(wgt, v.y, acc.y);
        acc.z = fmaf(wgt, v.z, acc.z);
        acc.w = fmaf(wgt, v.w, acc.w);
        wsum += wgt;
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    if (p.o_f32 != nullptr) {
      reinterpret_cast<float4*>(p.o_f32 + ((int64_t)tok * p.Hq + h) * D)[e4] =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      uint2 packed;
      packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.o) + ((int64_t)tok * p.Hq + h) * D)[e4] = packed;
    }
    if (e4 == 0 && p.lse != nullptr) p.lse[(int64_t)tok * p.Hq + h] = wsum > 0.f ? (mx + __log2f(wsum)) * kLn2 : -INFINITY;
  }
}

// Merge of partial states: grid (row, block of 128 (head, 4-column) items), one item per thread
// (bf16 output, or fp32 when o_f32 is set):
//   lse = log sum_p exp(lse_p),  O = sum_p exp(lse_p - lse) O_p.
// A part with lse_p = -inf has no keys; its O_p is never read (it may hold any bits). The loop over
// parts is unrolled so several parts' loads are in flight at once.
template <bool LOG2>
__global__ void __launch_bounds__(128) merge_kernel(const float* __restrict__ o_part,
                                                    const float* __restrict__ lse_part, int num_parts, int n_rows,
                                                    int H, int D, __nv_bfloat16* __restrict__ o,
                                                    float* __restrict__ o_f32, float* __restrict__ lse) {
  griddep_wait();  // launched as a programmatic dependent: the partial states must be complete
  const int64_t row = blockIdx.x;
  const int per_head = D / 4;
  const int t = blockIdx.y * blockDim.x + threadIdx.x;
  if (t >= H * per_head) return;
  const int h = t / per_head, e4 = t % per_head;
  const int64_t lrow = row * H + h;                // (row, head) in one part
  const int64_t pstride = (int64_t)n_rows * H;     // rows x heads of one part
  float mx = -INFINITY;
  for (int s = 0; s < num_parts; ++s) mx = fmaxf(mx, __ldg(&lse_part[s * pstride + lrow]));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (mx != -INFINITY) {
#pragma unroll 4
    for (int s = 0; s < num_parts; ++s) {
      const float ls = __ldg(&lse_part[s * pstride + lrow]);
      if (ls == -INFINITY) continue;
      const float w = LOG2 ? ex2(ls - mx) : __expf(ls - mx);
      const float4 v = __ldg(reinterpret_cast<const float4*>(o_part + (s * pstride + lrow) * D) + e4);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
      wsum += w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  if (o_f32 != nullptr) {
    reinterpret_cast<float4*>(o_f32 + lrow * D)[e4] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  } else {
    uint2 packed;
    packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2*>(o + lrow * D)[e4] = packed;
  }
  if (e4 == 0 && lse != nullptr) {
    float out = -INFINITY;
    if (wsum > 0.f) out = LOG2 ? (mx + __log2f(wsum)) * kLn2 : mx + __logf(wsum);
    lse[lrow] = out;
  }
}

template <int D, int G>
cudaError_t launch_decode_impl(const DecodeParams& p, cudaStream_t stream) {
  auto kern = decode_kernel<D, G>;
  const int chunk = kRowsPerBlock * p.heads_per_cta * D * 2;
  int n_stages = (200 * 1024) / (2 * chunk);
  n_stages = max(2, min(8, n_stages));
  const int smem = 128 + n_stages * 2 * chunk;
  // largest dynamic smem already allowed, per device (atomics: calls may come from several threads)
  static std::atomic<int> configured_smem[32];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 32 || configured_smem[dev].load(std::memory_order_acquire) < smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < 32) {
      int seen = configured_smem[dev].load(std::memory_order_relaxed);
      while (seen < smem && !configured_smem[dev].compare_exchange_weak(seen, smem, std::memory_order_release)) {
      }
    }
  }
  if (p.num_seqs > kDecodeMaxSeqs || p.Hkv / p.heads_per_cta > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(p.num_splits, p.num_seqs, p.Hkv / p.heads_per_cta);
  if (p.num_splits > 1) {
    // arrival counters of the fused merge start at zero on every call
    cudaError_t e = cudaMemsetAsync(p.counters, 0, sizeof(int) * (size_t)p.num_seqs * (p.Hkv / p.heads_per_cta),
                                    stream);
    if (e != cudaSuccess) return e;
  }
  kern<<<grid, p.heads_per_cta * 32, smem, stream>>>(p, n_stages);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t stream) {
  if (d == 128) {
    switch (p.group) {
      case 1: return launch_decode_impl<128, 1>(p, stream);
      case 2: return launch_decode_impl<128, 2>(p, stream);
      case 4: return launch_decode_impl<128, 4>(p, stream);
      case 8: return launch_decode_impl<128, 8>(p, stream);
    }
  } else {
    switch (p.group) {
      case 1: return launch_decode_impl<64, 1>(p, stream);
      case 2: return launch_decode_impl<64, 2>(p, stream);
      case 4: return launch_decode_impl<64, 4>(p, stream);
      case 8: return launch_decode_impl<64, 8>(p, stream);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_merge(const float* o_part, const float* lse_part, int num_parts, int n_rows, int H, int d, void* o,
                         float* o_f32, float* lse, bool log2_domain, cudaStream_t stream, bool programmatic) {
  auto* ob = reinterpret_cast<__nv_bfloat16*>(o);
  const dim3 grid((unsigned)n_rows, (unsigned)((H * (d / 4) + 127) / 128));
  if (programmatic) {
    // the CTAs may be resident before the kernel ahead of them ends; they wait for it first
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return log2_domain ? cudaLaunchKernelEx(&cfg, merge_kernel<true>, o_part, lse_part, num_parts, n_rows, H, d, ob,
                                            o_f32, lse)
                       : cudaLaunchKernelEx(&cfg, merge_kernel<false>, o_part, lse_part, num_parts, n_rows, H, d, ob,
                                            o_f32, lse);
  }
  if (log2_domain)
    merge_kernel<true><<<grid, 128, 0, stream>>>(o_part, lse_part, num_parts, n_rows, H, d, ob, o_f32, lse);
  else
    merge_kernel<false><<<grid, 128, 0, stream>>>(o_part, lse_part, num_parts, n_rows, H, d, ob, o_f32, lse);
  return cudaGetLastError();
}

}  // namespace fa
