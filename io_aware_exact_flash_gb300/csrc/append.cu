// Paged KV append: the key and value rows of new tokens written into their page slots.
//
// "I/O-Aware Kernels" (datasystem.school, Module 5), section "FlashInfer: I/O-aware attention
// for serving": the KV cache of a serving batch lives in fixed-size pages reached through a page
// table, so a sequence grows by writing each new token's rows into the slot after its current
// length, in whichever physical page the table names for that position.
//
// One token's K row is [Hkv, d] bf16, contiguous both in the packed input and in its page slot,
// so the append is a set of independent contiguous copies of Hkv * d * 2 bytes (K) plus the same
// for V: pure HBM traffic (read once, written once). One warp moves one token; each lane keeps up
// to 4 + 4 sixteen-byte loads in flight before it stores, and the grid is a multiple of the SM
// count with a grid-stride loop over tokens.
#include <cuda_runtime.h>
#include <cstdint>
#include "../../include/fa.h"
#include "kernels.cuh"

namespace {

using fa::DeviceStatus;

// Token t of sequence s (cu_seqlens_new[s] <= t < cu_seqlens_new[s + 1]) goes to logical
// position kv_lens_before[s] + (t - cu_seqlens_new[s]) of that sequence.
struct AppendParams {
  const void* k_new;               // [total_new, Hkv, d] bf16
  const void* v_new;
  const int32_t* cu_seqlens_new;   // [num_seqs + 1]
  const int32_t* kv_lens_before;   // [num_seqs]
  const int32_t* page_table;       // [num_seqs, max_pages_per_seq]
  void* k_pages;                   // [num_pages, page_size, Hkv, d] bf16, written in place
  void* v_pages;
  int64_t total_new;
  int num_seqs, page_size, max_pages_per_seq, num_pages;
  int row_vec16;                   // Hkv * d * 2 / 16
  DeviceStatus* status;
};

constexpr int kAppendThreads = 256;
constexpr int kAppendUnroll = 4;
enum : uint32_t { kSiteAppendBadPage = 24 };

__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }

__global__ void __launch_bounds__(kAppendThreads) append_kernel(AppendParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kAppendThreads / 32);
  const int n16 = p.row_vec16;  // 16-byte vectors per token row of K (and of V)
  for (int64_t t = (int64_t)blockIdx.x * (kAppendThreads / 32) + threadIdx.x / 32; t < p.total_new; t += warps) {
    // sequence of token t: the s with cu_new[s] <= t < cu_new[s + 1] (the interval halves every
    // step, so the search ends after log2(num_seqs) steps whatever the array holds)
    int lo = 0, hi = p.num_seqs;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(&p.cu_seqlens_new[mid]) <= t) lo = mid; else hi = mid;
    }
    const int64_t r = t - __ldg(&p.cu_seqlens_new[lo]);
    if (r < 0 || t >= __ldg(&p.cu_seqlens_new[lo + 1])) continue;  // token outside every sequence
    const int64_t pos = (int64_t)__ldg(&p.kv_lens_before[lo]) + r;
    const int64_t lp = pos / p.page_size;
    int page = -1;
    if (pos >= 0 && lp < p.max_pages_per_seq) page = __ldg(&p.page_table[(int64_t)lo * p.max_pages_per_seq + lp]);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) {
        atomicCAS(&p.status->code, 0u, 8u /* FA_ERR_DEVICE_BAD_PAGE */);
        atomicExch(&p.status->where, kSiteAppendBadPage);
      }
      continue;
    }
    const int64_t slot = (int64_t)page * p.page_size + (pos - lp * p.page_size);
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_new) + t * n16;
    const uint4* vs = reinterpret_cast<const uint4*>(p.v_new) + t * n16;
    uint4* kd = reinterpret_cast<uint4*>(p.k_pages) + slot * n16;
    uint4* vd = reinterpret_cast<uint4*>(p.v_pages) + slot * n16;
    for (int i0 = 0; i0 < n16; i0 += 32 * kAppendUnroll) {
      uint4 a[kAppendUnroll], b[kAppendUnroll];
#pragma unroll
      for (int u = 0; u < kAppendUnroll; ++u) {
        const int i = i0 + u * 32 + lane;
        if (i < n16) {
          a[u] = ld_stream(ks + i);
          b[u] = ld_stream(vs + i);
        }
      }
#pragma unroll
      for (int u = 0; u < kAppendUnroll; ++u) {
        const int i = i0 + u * 32 + lane;
        if (i < n16) {
          kd[i] = a[u];
          vd[i] = b[u];
        }
      }
    }
  }
}

bool aligned(const void* ptr, uintptr_t bytes) { return (reinterpret_cast<uintptr_t>(ptr) & (bytes - 1)) == 0; }

}  // namespace

extern "C" fa_status fa_paged_append(const void* k_new, const void* v_new, const int32_t* cu_seqlens_new,
                                     const int32_t* kv_lens_before, const int32_t* page_table, int num_seqs,
                                     int total_new, int page_size, int max_pages_per_seq, int num_pages, int Hkv,
                                     int d, void* k_pages, void* v_pages, fa_stream_t stream) {
  // with nothing to append the row buffers may be empty (NULL)
  if ((total_new > 0 && (!k_new || !v_new)) || !cu_seqlens_new || !kv_lens_before || !page_table || !k_pages ||
      !v_pages)
    return FA_ERR_INVALID_ARG;
  if (num_seqs <= 0 || total_new < 0 || page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0 || Hkv <= 0)
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)num_pages * page_size > (1LL << 31) - 1) return FA_ERR_UNSUPPORTED;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
      !aligned(cu_seqlens_new, 4) || !aligned(kv_lens_before, 4) || !aligned(page_table, 4))
    return FA_ERR_ALIGNMENT;
  DeviceStatus* status = nullptr;
  int sm_count = 0;
  const int dev_rc = fa::current_device_info(&status, &sm_count);
  if (dev_rc != FA_OK) return (fa_status)dev_rc;
  if (total_new == 0) return FA_OK;

  AppendParams p;
  p.k_new = k_new;
  p.v_new = v_new;
  p.cu_seqlens_new = cu_seqlens_new;
  p.kv_lens_before = kv_lens_before;
  p.page_table = page_table;
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.total_new = total_new;
  p.num_seqs = num_seqs;
  p.page_size = page_size;
  p.max_pages_per_seq = max_pages_per_seq;
  p.num_pages = num_pages;
  p.row_vec16 = Hkv * d * 2 / 16;
  p.status = status;
  int64_t blocks = ((int64_t)total_new + kAppendThreads / 32 - 1) / (kAppendThreads / 32);
  const int64_t cap = (int64_t)sm_count * 8;  // 8 resident CTAs of 256 threads per SM
  if (blocks > cap) blocks = cap;
  append_kernel<<<(unsigned)blocks, kAppendThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
