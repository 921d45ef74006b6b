// Split-KV paged decode that needs no workspace from its caller.
//
// fa_paged_fwd asks the caller for a device workspace to hold the per-split partial outputs and
// LSEs of split-KV decode. Some callers cannot provide one: they run where they may not call
// cudaMalloc (an engine that hands all device memory to a fixed arena up front, a plugin inside
// a host that owns every allocation, a serving loop that must never enter the allocator), and
// they have no spare buffer to lend. fa_paged_decode_noalloc serves them with scratch that is
// part of this library's device image: a fixed array of kNoAllocScratchBytes bytes that every
// GPU which loads the library keeps until the process exits. The caller still passes its inputs
// and outputs; this file allocates and frees nothing.
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include "../../include/fa.h"
#include "kernels.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = FA_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes == (size_t)16 << 20, "header and library disagree on the scratch size");

// The shared scratch: partial O values, partial LSEs and the merge's arrival counters.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

size_t partials_bytes(int splits, int num_seqs, int Hq, int Hkv, int d) {
  return fa::decode_scratch_bytes(splits, num_seqs, Hq, Hkv, d);
}

// Device address of the scratch on the current device. The host-side name of a __device__
// array is only a stand-in, so the address is looked up once per device with that device
// current and cached.
fa_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_paged_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                             const int32_t* page_table, const int32_t* cu_seqlens_q,
                                             const int32_t* kv_lens, int num_seqs, int total_q, int page_size,
                                             int max_pages_per_seq, int num_pages, int Hq, int Hkv, int d,
                                             float scale, void* o, float* lse, int num_splits,
                                             fa_stream_t stream) {
  if (!q || !k_pages || !v_pages || !page_table || !cu_seqlens_q || !kv_lens || !o) return FA_ERR_INVALID_ARG;
  if (num_seqs <= 0 || total_q < 0 || page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0 || Hq <= 0 ||
      Hkv <= 0 || Hq % Hkv != 0 || num_splits < 0 || !std::isfinite(scale) || !(scale > 0.f))
    return FA_ERR_INVALID_ARG;
  // decode only: every sequence has at most one query row, so there are at most num_seqs rows
  if (total_q > num_seqs) return FA_ERR_INVALID_ARG;
  if (num_seqs > fa::kDecodeMaxSeqs) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) return FA_ERR_UNSUPPORTED;
  const int group = Hq / Hkv;
  if (group != 1 && group != 2 && group != 4 && group != 8) return FA_ERR_UNSUPPORTED;
  if ((long long)max_pages_per_seq * page_size > (1LL << 30) || (long long)num_pages * page_size > (1LL << 31) - 1)
    return FA_ERR_UNSUPPORTED;
  auto misaligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (misaligned(q, 16) || misaligned(k_pages, 16) || misaligned(v_pages, 16) || misaligned(o, 16) ||
      (lse && misaligned(lse, 4)) || misaligned(page_table, 4) || misaligned(cu_seqlens_q, 4) ||
      misaligned(kv_lens, 4))
    return FA_ERR_ALIGNMENT;

  // A split count never exceeds the pages of the longest sequence. An explicit count whose
  // partials do not fit the scratch (after that cap) is rejected; the automatic count is lowered
  // until they fit (one split needs no scratch at all).
  int splits = num_splits > 0 ? num_splits : fa_decode_num_splits(num_seqs, page_size, max_pages_per_seq, num_pages, Hkv);
  if (splits > max_pages_per_seq) splits = max_pages_per_seq;
  if (splits < 1) splits = 1;
  if (num_splits > 0) {
    if (partials_bytes(splits, num_seqs, Hq, Hkv, d) > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  } else {
    while (splits > 1 && partials_bytes(splits, num_seqs, Hq, Hkv, d) > kNoAllocScratchBytes) --splits;
  }

  fa::DeviceStatus* status = nullptr;
  int sm_count = 0;
  const int dev_rc = fa::current_device_info(&status, &sm_count);
  if (dev_rc != FA_OK) return static_cast<fa_status>(dev_rc);
  void* scratch = nullptr;
  const fa_status s_rc = scratch_on_current_device(&scratch);
  if (s_rc != FA_OK) return s_rc;
  if (total_q == 0) return FA_OK;

  fa::DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.page_table = page_table;
  p.cu_seqlens_q = cu_seqlens_q;
  p.kv_lens = kv_lens;
  p.o = o;
  p.lse = lse;
  if (splits > 1) fa::decode_scratch_layout(scratch, splits, num_seqs, Hq, d, p);
  p.num_seqs = num_seqs;
  p.total_q = total_q;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = group;
  p.page_size = page_size;
  p.max_pages_per_seq = max_pages_per_seq;
  p.num_pages = num_pages;
  p.num_splits = splits;
  p.pages_per_split = (max_pages_per_seq + splits - 1) / splits;
  p.heads_per_cta = fa::decode_heads_per_cta(Hkv);
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.status = status;
  return fa::launch_decode(p, d, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
