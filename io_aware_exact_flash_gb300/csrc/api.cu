// C ABI of the attention library (declared in include/fa.h): argument validation, TMA tensor
// descriptors, work planning and kernel dispatch. Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include "../../include/fa.h"
#include "kernels.cuh"

// The one piece of global device state: a status word per GPU that kernels set instead of
// trapping (a wait that timed out, a page id outside the pool).
__device__ fa::DeviceStatus g_fa_device_status;

namespace {

using fa::DeviceStatus;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool probed = false;
  bool supported = false;
  int sm_count = 0;
  DeviceStatus* status = nullptr;  // device address of g_fa_device_status on this GPU
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Looks up (once per GPU) whether the current device is an sm_103 part, its SM count and the
// device address of the status word. Returns nullptr on failure.
const DeviceInfo* current_device(fa_status* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = FA_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& info = g_dev[dev];
  if (!info.probed) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      *err = FA_ERR_CUDA;
      return nullptr;
    }
    info.supported = (prop.major == 10 && prop.minor == 3);
    info.sm_count = prop.multiProcessorCount;
    void* addr = nullptr;
    if (info.supported) {
      if (cudaGetSymbolAddress(&addr, g_fa_device_status) != cudaSuccess) {
        *err = FA_ERR_CUDA;
        return nullptr;
      }
    }
    info.status = static_cast<DeviceStatus*>(addr);
    info.probed = true;
  }
  if (!info.supported) {
    *err = FA_ERR_NO_DEVICE;
    return nullptr;
  }
  return &info;
}

// cuTensorMapEncodeTiled, fetched from the driver once (no link-time dependency on libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 4-D bf16 tensor map with 128-byte swizzle; dims innermost first, strides in bytes for dims 1..3.
bool make_map(CUtensorMap* m, const void* base, const uint64_t dims[4], const uint64_t strides[3],
              const uint32_t box[4]) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t gs[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t bd[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gd, gs, bd, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- paged planning helpers
struct DecodePlan {
  int splits;
  int pages_per_split;
  int heads_per_cta;
};

DecodePlan plan_decode(int num_seqs, int page_size, int max_pages_per_seq, int num_pages, int Hkv, int num_splits,
                       int sm_count) {
  DecodePlan d;
  d.heads_per_cta = fa::decode_heads_per_cta(Hkv);
  const int head_blocks = Hkv / d.heads_per_cta;
  int splits = num_splits;
  if (splits <= 0) {
    // Aim for about eight CTAs per SM over the whole batch: the pool holds about num_pages pages
    // in use, and the longest sequence sets how many splits are needed to cut it that finely.
    const long long target_ctas = 8LL * (sm_count > 0 ? sm_count : 148);
    const long long work_pages = (long long)(num_pages > 0 ? num_pages : num_seqs) * head_blocks;
    long long pps = (work_pages + target_ctas - 1) / target_ctas;
    if (pps < 1) pps = 1;
    splits = (int)((max_pages_per_seq + pps - 1) / pps);
    if (splits < 1) splits = 1;
    if (splits > 256) splits = 256;
  }
  if (splits > max_pages_per_seq) splits = max_pages_per_seq > 0 ? max_pages_per_seq : 1;
  d.splits = splits;
  d.pages_per_split = (max_pages_per_seq + splits - 1) / splits;
  if (d.pages_per_split < 1) d.pages_per_split = 1;
  return d;
}

// Work items (tile pairs) of a paged prefill launch are at most total_q * pack / 256 + num_seqs.
int prefill_max_items(int num_seqs, int total_q, int pack) {
  return (int)((long long)total_q * pack / 256) + num_seqs;
}

size_t decode_workspace(int num_seqs, int Hq, int Hkv, int d, int splits) {
  return fa::decode_scratch_bytes(splits, num_seqs, Hq, Hkv, d);
}

// count | work list (int2 per item) | sequence order and item offsets (2 ints per sequence)
size_t prefill_workspace(int num_seqs, int total_q, int pack) {
  return 256 + align_up((size_t)prefill_max_items(num_seqs, total_q, pack) * sizeof(int2) +
                            2 * sizeof(int) * num_seqs,
                        256);
}

int sm_count_now() {
  fa_status e;
  const DeviceInfo* info = current_device(&e);
  if (info) return info->sm_count;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
    return n;
  return 148;
}

// Diagnostic: one warp waits on an mbarrier phase that nothing will ever complete. The bounded
// wait must give up after limit_ns, record FA_ERR_DEVICE_TIMEOUT with the site id in the status
// word and let the kernel exit normally.
constexpr uint32_t kSiteSelftest = 99;

__global__ void wait_timeout_selftest_kernel(DeviceStatus* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    fa::mbar_init(&bar, 1);
    fa::fence_mbar_init();
  }
  __syncthreads();
  fa::mbar_wait(&bar, 0, &abort_flag, status, kSiteSelftest, limit_ns);
}

}  // namespace

int fa::current_device_info(DeviceStatus** status, int* sm_count) {
  fa_status err = FA_OK;
  const DeviceInfo* dev = current_device(&err);
  if (!dev) return err;
  *status = dev->status;
  *sm_count = dev->sm_count;
  return FA_OK;
}

namespace {

// Shape checks shared by fa_paged_fwd and the two passes of fa_cascade_fwd.
fa_status check_paged_shape(int num_seqs, int total_q, int max_q_len, int page_size, int max_pages_per_seq,
                            int num_pages, int Hq, int Hkv, int d, int num_splits, float scale) {
  if (num_seqs <= 0 || total_q < 0 || max_q_len < 1 || page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0 ||
      Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_splits < 0 || !scale_ok(scale))
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)max_pages_per_seq * page_size > (1LL << 30) || (long long)num_pages * page_size > (1LL << 31) - 1)
    return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Reads a 0/1 switch from the environment once; -1 when it is unset or holds anything else.
int env_switch(const char* name, std::atomic<int>* cache) {
  int v = cache->load(std::memory_order_relaxed);
  if (v == -2) {
    const char* e = getenv(name);
    v = (e == nullptr || (e[0] != '0' && e[0] != '1') || e[1] != '\0') ? -1 : (e[0] == '1');
    cache->store(v, std::memory_order_relaxed);
  }
  return v;
}

bool pow2_group(int group) { return group >= 2 && group <= fa::kBM && (group & (group - 1)) == 0; }

// GQA packing of the paged tensor-core path: the query heads that share a kv head fill one tile
// together (rows = token x head, 128 / group tokens), so every K/V tile is read once for the
// whole group and sequences with few query tokens (multi-token verify, decode rows of a mixed
// batch) fill their tiles instead of holding a handful of rows. Measured faster on every paged
// workload with group 4 (long ragged prefill +3%, mixed batch +15%, verify 3.7x), so it is the
// default for every power-of-two group up to 128 (MQA included). FA_PAGED_PACK=0 turns it off.
int choose_pack(int group, int max_q_len) {
  (void)max_q_len;
  if (!pow2_group(group)) return 1;
  static std::atomic<int> mode{-2};
  return env_switch("FA_PAGED_PACK", &mode) == 0 ? 1 : group;
}

// Decode batches (one query row per sequence) run on the tensor-core path: with a packed group a
// tile holds every query head of a kv head, and in any case the MMAs cost far less than streaming
// the keys, so the path is bound by reading K/V. Measured against the split-KV CUDA-core kernel:
// group 4, 128 sequences 5410 vs 4683 GB/s, 32 sequences 3999 vs 3097; MHA (group 1, one real
// row per tile), 32 sequences 5501 vs 4501. FA_DECODE_TC=0 sends groups 1, 2, 4 and 8 (the
// groups that kernel takes) to the CUDA-core kernel.
bool decode_on_tensor_cores(int group) {
  static std::atomic<int> mode{-2};
  if (group == 1 || group == 2 || group == 4 || group == 8) return env_switch("FA_DECODE_TC", &mode) != 0;
  return true;
}

// Batches whose sequences have at most 16 query rows per kv head (decode up to group 16, verify of
// a few tokens) at d = 128 run on the key-row kernel (decode_tc.cu): the keys of a tile are the
// MMA's 128 rows and the query rows its columns. Measured against the packed prefill kernel on the
// decode workload (128 sequences, group 4): 0.660 against 0.763 ms; 16 sequences with 4 key
// splits 0.094 against 0.112 ms; the cascade (its suffix pass) 0.169 against 0.198 ms. Batches
// of more rows per kv head (verify of 5-8 tokens at group 4) stay on the packed kernel: a 32-column
// form of the key-row kernel measured 0.77 against 0.81 ms there, but needs a second softmax
// warpgroup, and 13 warps leave 128 registers a thread (it spilled). FA_DECODE_KEY_ROWS=0 sends
// every batch to the packed kernel.
int key_row_max_rows() {
  static std::atomic<int> mode{-2};
  return env_switch("FA_DECODE_KEY_ROWS", &mode) == 0 ? 0 : 16;
}

// Key splits of the paged tensor-core path. Each (tile pair, head slot) unit becomes kv_splits
// units over contiguous key ranges, written as fp32 partial states and merged by their LSE
// afterwards. Splitting pays when there are too few units to fill the GPU a few times over
// (small decode batches, one long shared prefix); each split keeps at least 8 key tiles, and
// the partial states are kept under 1 GiB. (Targets of 2, 3, 4 and 6 waves with at least 4 or 8
// tiles were measured on decode batches of 4 to 64 sequences and the cascade; 3 and 8 was best
// or level everywhere.) Units whose two query tiles are full (a shared prefix seen by many query
// rows) are compute bound instead, and there whole waves matter: the count with the shortest
// estimated makespan, waves x (key tiles per split + a per-unit cost of kSplitUnitCostTiles key
// tiles: loads, epilogue, partial state), is taken. On the cascade's prefix (16 units over 128
// key tiles) that is 9 splits, one wave, 60 us, against 16 splits, 1.7 waves, 73 us (the per-unit
// cost was fitted to a sweep of 4 to 24 splits there). requested > 0 fixes the count (capped at
// the key tiles of the longest sequence).
constexpr int kSplitUnitCostTiles = 6;
int plan_kv_splits(int num_seqs, int total_q, int max_q_len, int pack, int Hq, int d, int max_kv_tiles,
                   int sm_count, int requested) {
  if (max_kv_tiles < 1) max_kv_tiles = 1;
  if (requested > 0) return requested < max_kv_tiles ? requested : max_kv_tiles;
  const long long pairs_per_seq = ((long long)max_q_len * pack + 2 * fa::kBM - 1) / (2 * fa::kBM);
  long long items = (long long)num_seqs * pairs_per_seq;
  const long long bound = prefill_max_items(num_seqs, total_q, pack);
  if (items > bound) items = bound;
  const long long units = items * (Hq / pack);
  const long long target = 3LL * sm_count;
  if (units <= 0 || units >= target) return 1;
  long long s_max = max_kv_tiles / 8;
  const long long part = (long long)total_q * Hq * (d + 1) * 4;
  if (part > 0 && s_max * part > (1LL << 30)) s_max = (1LL << 30) / part;
  if (s_max < 1) return 1;
  long long s;
  if ((long long)max_q_len * pack >= 2 * fa::kBM) {
    s = 1;
    long long best = -1;
    for (long long c = 1; c <= s_max; ++c) {
      const long long waves = (units * c + sm_count - 1) / sm_count;
      const long long cost = waves * ((max_kv_tiles + c - 1) / c + kSplitUnitCostTiles);
      if (best < 0 || cost < best) {
        best = cost;
        s = c;
      }
    }
  } else {
    s = (target + units - 1) / units;
    if (s > s_max) s = s_max;
  }
  return s < 1 ? 1 : (int)s;
}

// fp32 partial states of a split tensor-core pass: O parts then LSE parts, each 256-byte aligned.
size_t split_parts_bytes(int kv_splits, int total_q, int Hq, int d, size_t* lse_offset) {
  if (kv_splits <= 1) {
    if (lse_offset) *lse_offset = 0;
    return 0;
  }
  const size_t o_bytes = align_up((size_t)kv_splits * total_q * Hq * d * sizeof(float), 256);
  if (lse_offset) *lse_offset = o_bytes;
  return o_bytes + align_up((size_t)kv_splits * total_q * Hq * sizeof(float), 256);
}

int max_kv_tiles_of(int max_pages_per_seq, int page_size) {
  long long t = ((long long)max_pages_per_seq * page_size + fa::kBN - 1) / fa::kBN;
  return (int)(t > (1 << 30) ? (1 << 30) : t);
}

// Workspace of one paged pass (decode partials, or the prefill work list).
// The key-split count of one paged pass (1 on the CUDA-core decode kernel, which merges its own).
int paged_pass_splits(int num_seqs, int total_q, int max_q_len, int page_size, int max_pages_per_seq, int Hq, int Hkv,
                      int d, int num_splits, int sm_count) {
  const int group = Hkv > 0 ? Hq / Hkv : 0;
  if (max_q_len == 1 && !decode_on_tensor_cores(group)) return 1;
  return plan_kv_splits(num_seqs, total_q, max_q_len, choose_pack(group, max_q_len), Hq, d,
                        max_kv_tiles_of(max_pages_per_seq, page_size), sm_count, num_splits);
}

// Workspace of one paged pass. external_parts: the pass writes its split partial states into the
// caller's part arrays (no merge of its own), so they are not counted here.
size_t paged_pass_workspace(int num_seqs, int total_q, int max_q_len, int page_size, int max_pages_per_seq,
                            int num_pages, int Hq, int Hkv, int d, int num_splits, int sm_count,
                            bool external_parts = false) {
  const int group = Hkv > 0 ? Hq / Hkv : 0;
  if (max_q_len == 1 && !decode_on_tensor_cores(group)) {
    const DecodePlan dp = plan_decode(num_seqs, page_size, max_pages_per_seq, num_pages, Hkv, num_splits, sm_count);
    return decode_workspace(num_seqs, Hq, Hkv, d, dp.splits);
  }
  const int pack = choose_pack(group, max_q_len);
  const int splits = plan_kv_splits(num_seqs, total_q, max_q_len, pack, Hq, d,
                                    max_kv_tiles_of(max_pages_per_seq, page_size), sm_count, num_splits);
  return prefill_workspace(num_seqs, total_q, pack) +
         (external_parts ? 0 : split_parts_bytes(splits, total_q, Hq, d, nullptr));
}

// Enqueue one validated paged pass. O goes to `o` as bf16, or to `o_f32` as fp32 when that is set.
fa_status enqueue_paged(const DeviceInfo* dev, const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* page_table, const int32_t* cu_seqlens_q, const int32_t* kv_lens, int num_seqs,
                        int total_q, int max_q_len, int page_size, int max_pages_per_seq, int num_pages, int Hq,
                        int Hkv, int d, int causal, float scale, void* o, float* o_f32, float* lse, void* workspace,
                        size_t workspace_bytes, int num_splits, fa_stream_t stream, float* ext_o_parts = nullptr,
                        float* ext_lse_parts = nullptr, cudaEvent_t after_plan = nullptr) {
  // after_plan: recorded once the pass's planning kernel is queued (or, on a path without one,
  // before its first launch), so that other streams can start work that must not run ahead of
  // this pass taking its SMs
  if (total_q == 0) return after_plan && cudaEventRecord(after_plan, stream) != cudaSuccess ? FA_ERR_CUDA : FA_OK;
  const int group = Hq / Hkv;

  if (max_q_len == 1 && !decode_on_tensor_cores(group)) {
    // ------------------------------------------------------------- split-KV decode
    if (group != 1 && group != 2 && group != 4 && group != 8) return FA_ERR_UNSUPPORTED;
    if (num_seqs > fa::kDecodeMaxSeqs) return FA_ERR_UNSUPPORTED;
    const DecodePlan dp =
        plan_decode(num_seqs, page_size, max_pages_per_seq, num_pages, Hkv, num_splits, dev->sm_count);
    const size_t need = decode_workspace(num_seqs, Hq, Hkv, d, dp.splits);
    if (need > 0 && (!workspace || workspace_bytes < need)) return FA_ERR_WORKSPACE;
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FA_ERR_ALIGNMENT;
    fa::DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q;
    p.k_pages = k_pages;
    p.v_pages = v_pages;
    p.page_table = page_table;
    p.cu_seqlens_q = cu_seqlens_q;
    p.kv_lens = kv_lens;
    p.o = o;
    p.o_f32 = o_f32;
    p.lse = lse;
    if (need > 0) fa::decode_scratch_layout(workspace, dp.splits, num_seqs, Hq, d, p);
    p.num_seqs = num_seqs;
    p.total_q = total_q;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = group;
    p.page_size = page_size;
    p.max_pages_per_seq = max_pages_per_seq;
    p.num_pages = num_pages;
    p.pages_per_split = dp.pages_per_split;
    p.num_splits = dp.splits;
    p.heads_per_cta = dp.heads_per_cta;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.status = dev->status;
    if (after_plan && cudaEventRecord(after_plan, stream) != cudaSuccess) return FA_ERR_CUDA;
    return fa::launch_decode(p, d, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }

  // --------------------------------------------------------------- tensor-core path
  const int pack = choose_pack(group, max_q_len);
  const int max_kv_tiles = max_kv_tiles_of(max_pages_per_seq, page_size);
  const int kv_splits =
      plan_kv_splits(num_seqs, total_q, max_q_len, pack, Hq, d, max_kv_tiles, dev->sm_count, num_splits);
  // units (tile pairs x head slots x key splits) are counted in 32-bit integers on the device
  if ((long long)prefill_max_items(num_seqs, total_q, pack) * (Hq / pack) * kv_splits >= (1LL << 31))
    return FA_ERR_UNSUPPORTED;
  const size_t list_bytes = prefill_workspace(num_seqs, total_q, pack);
  // ext_o_parts: split partial states go to the caller's part arrays, which it merges itself
  const bool external = ext_o_parts != nullptr && kv_splits > 1;
  size_t lse_off = 0;
  const size_t need = list_bytes + (external ? 0 : split_parts_bytes(kv_splits, total_q, Hq, d, &lse_off));
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGNMENT;
  // batches of a few query rows per (sequence, kv head) run with the keys on the MMA's rows
  const int kr_columns = fa::decode_tc_columns(max_q_len, group, d, key_row_max_rows());
  fa::PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  {
    // a Q tile is `pack` heads x (128 / pack) tokens: with pack > 1, row r of the tile is token
    // r / pack and head r % pack of the box (the box's inner dimensions are d, then heads). On
    // the key-row path a unit's Q rows are the group's heads x (columns / group) tokens.
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)Hq, (uint64_t)total_q, 1};
    const uint64_t str[3] = {(uint64_t)d * 2, (uint64_t)Hq * d * 2, (uint64_t)total_q * Hq * d * 2};
    const uint32_t box[4] = {64, (uint32_t)(kr_columns > 0 ? group : pack),
                             (uint32_t)(kr_columns > 0 ? 16 / group : fa::kBM / pack), 1};
    if (!make_map(&p.tm_q, q, dims, str, box)) return FA_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)Hkv, (uint64_t)page_size, (uint64_t)num_pages};
    const uint64_t str[3] = {(uint64_t)d * 2, (uint64_t)Hkv * d * 2, (uint64_t)page_size * Hkv * d * 2};
    const uint32_t box[4] = {64, 1, (uint32_t)page_size, 1};
    if (!make_map(&p.tm_k, k_pages, dims, str, box) || !make_map(&p.tm_v, v_pages, dims, str, box))
      return FA_ERR_CUDA;
  }
  int* work_count = static_cast<int*>(workspace);
  int2* work_list = reinterpret_cast<int2*>(static_cast<char*>(workspace) + 256);
  p.o = o;
  p.o_f32 = o_f32;
  p.lse = lse;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = group;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.page_table = page_table;
  p.cu_seqlens_q = cu_seqlens_q;
  p.kv_lens = kv_lens;
  p.page_size = page_size;
  p.max_pages_per_seq = max_pages_per_seq;
  p.num_pages = num_pages;
  p.num_seqs = num_seqs;
  p.total_q = total_q;
  p.work_list = work_list;
  p.work_count = work_count;
  p.pack = pack;
  p.kv_splits = kv_splits;
  if (external) {
    p.o_part = ext_o_parts;
    p.lse_part = ext_lse_parts;
  } else if (kv_splits > 1) {
    char* parts = static_cast<char*>(workspace) + list_bytes;
    p.o_part = reinterpret_cast<float*>(parts);
    p.lse_part = reinterpret_cast<float*>(parts + lse_off);
  }
  p.status = dev->status;
  const int cost_buckets = max_kv_tiles > 8192 ? 8192 : max_kv_tiles;  // buckets only order the work
  if (kr_columns > 0) {
    // one planning item per sequence (at most 32 query rows); the unit's heads are the group
    p.pack = 1;
    if (fa::launch_decode_tc(p, kr_columns, dev->sm_count, prefill_max_items(num_seqs, total_q, pack), cost_buckets,
                             work_list, work_count, stream, after_plan) != cudaSuccess)
      return FA_ERR_CUDA;
  } else if (fa::launch_prefill_paged(p, d, dev->sm_count, prefill_max_items(num_seqs, total_q, pack), cost_buckets,
                                      work_list, work_count, stream, after_plan) != cudaSuccess) {
    return FA_ERR_CUDA;
  }
  if (kv_splits > 1 && !external &&
      fa::launch_merge(p.o_part, p.lse_part, kv_splits, total_q, Hq, d, o, o_f32, lse, false, stream,
                       kr_columns > 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_NO_DEVICE: return "FA_ERR_NO_DEVICE";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
    case FA_ERR_DEVICE_BAD_PAGE: return "FA_ERR_DEVICE_BAD_PAGE";
  }
  return "FA_ERR_UNKNOWN";
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int S,
                 int d, int causal, float scale, fa_stream_t stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || Hq % Hkv != 0 || !scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)B * S > (1LL << 31) - 1 || (long long)B * S * Hq * d > (1LL << 40)) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FA_ERR_ALIGNMENT;
  fa_status err = FA_OK;
  const DeviceInfo* dev = current_device(&err);
  if (!dev) return err;

  fa::PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  const uint32_t box[4] = {64, 1, (uint32_t)fa::kBM, 1};
  {
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)Hq, (uint64_t)S, (uint64_t)B};
    const uint64_t str[3] = {(uint64_t)d * 2, (uint64_t)Hq * d * 2, (uint64_t)S * Hq * d * 2};
    if (!make_map(&p.tm_q, q, dims, str, box)) return FA_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)Hkv, (uint64_t)S, (uint64_t)B};
    const uint64_t str[3] = {(uint64_t)d * 2, (uint64_t)Hkv * d * 2, (uint64_t)S * Hkv * d * 2};
    if (!make_map(&p.tm_k, k, dims, str, box) || !make_map(&p.tm_v, v, dims, str, box)) return FA_ERR_CUDA;
  }
  p.o = o;
  p.lse = lse;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.B = B;
  p.S = S;
  p.pack = 1;
  {
    // about one wave of CTAs per chunk of kv heads (see the unit order in prefill.cu)
    const long long per_kv_head = (long long)(Hq / Hkv) * ((S + 255) / 256);
    long long hc = (dev->sm_count + per_kv_head / 2) / per_kv_head;
    if (hc < 1) hc = 1;
    if (hc > (long long)B * Hkv) hc = (long long)B * Hkv;
    p.kv_heads_per_chunk = (int)hc;
  }
  p.status = dev->status;
  return fa::launch_prefill_dense(p, d, dev->sm_count, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_paged_num_splits(int num_seqs, int total_q, int max_q_len, int page_size, int max_pages_per_seq,
                        int num_pages, int Hq, int Hkv, int d) {
  if (check_paged_shape(num_seqs, total_q, max_q_len, page_size, max_pages_per_seq, num_pages, Hq, Hkv, d, 0, 1.f) !=
      FA_OK)
    return 1;
  const int group = Hq / Hkv;
  const int sms = sm_count_now();
  if (max_q_len == 1 && !decode_on_tensor_cores(group))
    return plan_decode(num_seqs, page_size, max_pages_per_seq, num_pages, Hkv, 0, sms).splits;
  return plan_kv_splits(num_seqs, total_q, max_q_len, choose_pack(group, max_q_len), Hq, d,
                        max_kv_tiles_of(max_pages_per_seq, page_size), sms, 0);
}

int fa_decode_num_splits(int num_seqs, int page_size, int max_pages_per_seq, int num_pages, int Hkv) {
  if (num_seqs <= 0 || page_size <= 0 || max_pages_per_seq <= 0 || Hkv <= 0) return 1;
  return plan_decode(num_seqs, page_size, max_pages_per_seq, num_pages, Hkv, 0, sm_count_now()).splits;
}

size_t fa_paged_workspace_bytes(int num_seqs, int total_q, int max_q_len, int page_size, int max_pages_per_seq,
                                int num_pages, int Hq, int Hkv, int d, int num_splits) {
  if (num_seqs <= 0 || total_q < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || page_size <= 0 || max_pages_per_seq <= 0)
    return 0;
  return paged_pass_workspace(num_seqs, total_q, max_q_len, page_size, max_pages_per_seq, num_pages, Hq, Hkv, d,
                              num_splits, sm_count_now());
}

fa_status fa_paged_fwd(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                       const int32_t* cu_seqlens_q, const int32_t* kv_lens, int num_seqs, int total_q, int max_q_len,
                       int page_size, int max_pages_per_seq, int num_pages, int Hq, int Hkv, int d, int causal,
                       float scale, void* o, float* lse, void* workspace, size_t workspace_bytes, int num_splits,
                       fa_stream_t stream) {
  if (!q || !k_pages || !v_pages || !page_table || !cu_seqlens_q || !kv_lens || !o) return FA_ERR_INVALID_ARG;
  fa_status err = check_paged_shape(num_seqs, total_q, max_q_len, page_size, max_pages_per_seq, num_pages, Hq, Hkv, d,
                                    num_splits, scale);
  if (err != FA_OK) return err;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) || (lse && !aligned4(lse)) ||
      !aligned4(page_table) || !aligned4(cu_seqlens_q) || !aligned4(kv_lens))
    return FA_ERR_ALIGNMENT;
  const DeviceInfo* dev = current_device(&err);
  if (!dev) return err;
  return enqueue_paged(dev, q, k_pages, v_pages, page_table, cu_seqlens_q, kv_lens, num_seqs, total_q, max_q_len,
                       page_size, max_pages_per_seq, num_pages, Hq, Hkv, d, causal, scale, o, nullptr, lse, workspace,
                       workspace_bytes, num_splits, stream);
}

// Shared-prefix (cascade) attention: the prefix pass leaves one fp32 partial state per key split
// (O normalised over its own keys, natural-log LSE), the suffix pass one more, and a single merge
// combines them all. Workspace: O parts [parts, total_q, Hq, d] fp32 | LSE parts [parts, total_q,
// Hq] fp32 | the passes' own scratch (reused by both, which run one after the other on the stream).
namespace {
// Key splits of the cascade's prefix pass. Its two passes run side by side (the suffix pass on a
// second stream): the prefix pass, bound by tensor work, takes a few SMs for longer while the
// suffix pass, bound by HBM, streams on the rest. A third of the split count that the pass would
// take alone leaves it about a third of the SMs; measured on 128 decode rows behind a
// 16384-token prefix (prefix splits, then side by side / one after the other, ms per call without
// the final merge): 2 splits 0.162 / 0.243, 3 splits 0.144 / 0.211, 4 0.145 / 0.193, 6 0.146 /
// 0.181, 9 (the pass alone's choice) 0.151 / 0.171.
int cascade_prefix_splits(int num_groups, int total_q, int max_group_q_len, int page_size, int max_prefix_pages,
                          int Hq, int Hkv, int d, int sm_count) {
  const int alone = paged_pass_splits(num_groups, total_q, max_group_q_len, page_size, max_prefix_pages, Hq, Hkv, d, 0,
                                      sm_count);
  return alone >= 3 ? alone / 3 : 1;
}

// The second stream and the fork / join events of the cascade, one set per host thread and GPU
// (created on first use, kept for the thread's lifetime). Null stream: run the passes in order.
struct SideStream {
  int device = -1;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
const SideStream* side_stream() {
  thread_local SideStream side[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& t = side[dev];
  if (t.device != dev) {
    t.device = dev;
    if (cudaStreamCreateWithFlags(&t.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&t.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&t.join, cudaEventDisableTiming) != cudaSuccess) {
      t.stream = nullptr;
      cudaGetLastError();  // leave no sticky error behind; the passes then run in order
    }
  }
  return t.stream ? &t : nullptr;
}

size_t cascade_parts_bytes(int parts, int total_q, int Hq, int d, size_t* lse_offset) {
  const size_t o_bytes = align_up((size_t)parts * total_q * Hq * d * sizeof(float), 256);
  if (lse_offset) *lse_offset = o_bytes;
  return o_bytes + align_up((size_t)parts * total_q * Hq * sizeof(float), 256);
}
}  // namespace

size_t fa_cascade_workspace_bytes(int num_groups, int num_seqs, int total_q, int max_group_q_len, int max_q_len,
                                  int page_size, int max_prefix_pages, int max_pages_per_seq, int num_pages, int Hq,
                                  int Hkv, int d) {
  if (check_paged_shape(num_groups, total_q, max_group_q_len, page_size, max_prefix_pages, num_pages, Hq, Hkv, d, 0,
                        1.f) != FA_OK ||
      check_paged_shape(num_seqs, total_q, max_q_len, page_size, max_pages_per_seq, num_pages, Hq, Hkv, d, 0, 1.f) !=
          FA_OK)
    return 0;
  const int sms = sm_count_now();
  const int sp =
      cascade_prefix_splits(num_groups, total_q, max_group_q_len, page_size, max_prefix_pages, Hq, Hkv, d, sms);
  const size_t a = paged_pass_workspace(num_groups, total_q, max_group_q_len, page_size, max_prefix_pages, num_pages,
                                        Hq, Hkv, d, sp, sms, true);
  const size_t b =
      paged_pass_workspace(num_seqs, total_q, max_q_len, page_size, max_pages_per_seq, num_pages, Hq, Hkv, d, 0, sms);
  // the passes may run side by side: each has a scratch region of its own
  return cascade_parts_bytes(sp + 1, total_q, Hq, d, nullptr) + align_up(a, 256) + b;
}

fa_status fa_cascade_fwd(const void* q, const void* k_pages, const void* v_pages, int page_size, int num_pages, int Hq,
                         int Hkv, int d, float scale, int num_groups, const int32_t* cu_q_groups,
                         const int32_t* prefix_page_table, const int32_t* prefix_lens, int max_prefix_pages,
                         int max_group_q_len, int num_seqs, const int32_t* cu_seqlens_q, const int32_t* page_table,
                         const int32_t* kv_lens, int max_pages_per_seq, int max_q_len, int causal, int total_q, void* o,
                         float* lse, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!q || !k_pages || !v_pages || !cu_q_groups || !prefix_page_table || !prefix_lens || !cu_seqlens_q ||
      !page_table || !kv_lens || !o)
    return FA_ERR_INVALID_ARG;
  fa_status err = check_paged_shape(num_groups, total_q, max_group_q_len, page_size, max_prefix_pages, num_pages, Hq,
                                    Hkv, d, 0, scale);
  if (err != FA_OK) return err;
  err = check_paged_shape(num_seqs, total_q, max_q_len, page_size, max_pages_per_seq, num_pages, Hq, Hkv, d, 0, scale);
  if (err != FA_OK) return err;
  if (num_groups > num_seqs) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) || (lse && !aligned4(lse)) ||
      !aligned4(cu_q_groups) || !aligned4(prefix_page_table) || !aligned4(prefix_lens) || !aligned4(cu_seqlens_q) ||
      !aligned4(page_table) || !aligned4(kv_lens))
    return FA_ERR_ALIGNMENT;
  const DeviceInfo* dev = current_device(&err);
  if (!dev) return err;
  if (total_q == 0) return FA_OK;
  const size_t need = fa_cascade_workspace_bytes(num_groups, num_seqs, total_q, max_group_q_len, max_q_len, page_size,
                                                 max_prefix_pages, max_pages_per_seq, num_pages, Hq, Hkv, d);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGNMENT;
  const int sp = cascade_prefix_splits(num_groups, total_q, max_group_q_len, page_size, max_prefix_pages, Hq, Hkv, d,
                                       dev->sm_count);
  size_t lse_off = 0;
  const size_t parts = cascade_parts_bytes(sp + 1, total_q, Hq, d, &lse_off);
  char* base = static_cast<char*>(workspace);
  float* o_parts = reinterpret_cast<float*>(base);
  float* lse_parts = reinterpret_cast<float*>(base + lse_off);
  const size_t part_rows = (size_t)total_q * Hq;
  // each pass plans into a scratch region of its own, so that they can run side by side
  const size_t scratch_a = align_up(paged_pass_workspace(num_groups, total_q, max_group_q_len, page_size,
                                                         max_prefix_pages, num_pages, Hq, Hkv, d, sp, dev->sm_count,
                                                         true),
                                    256);
  void* scratch_pre = base + parts;
  void* scratch_suf = base + parts + scratch_a;
  const size_t suf_bytes = workspace_bytes - parts - scratch_a;
  // The suffix pass runs on a second stream, forked from and joined back into `stream`. The fork
  // point is the prefix pass's planning kernel: the prefix's attention kernel is then queued before
  // the suffix's, takes its SMs first and runs beside the suffix pass, which fills the other SMs
  // and those the prefix frees. (Forked before the prefix's planning, the suffix's persistent grid
  // could take every SM first and push the prefix pass behind it.)
  const SideStream* side = side_stream();
  cudaStream_t suf_stream = stream;
  // prefix pass: every query row of a group sees all of the group's shared keys; its key splits
  // (parts 0 .. sp-1) are left for the final merge
  err = enqueue_paged(dev, q, k_pages, v_pages, prefix_page_table, cu_q_groups, prefix_lens, num_groups, total_q,
                      max_group_q_len, page_size, max_prefix_pages, num_pages, Hq, Hkv, d, 0, scale, nullptr, o_parts,
                      lse_parts, scratch_pre, scratch_a, sp, stream, sp > 1 ? o_parts : nullptr,
                      sp > 1 ? lse_parts : nullptr, side ? side->fork : nullptr);
  if (err == FA_OK && side) {
    if (cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess) return FA_ERR_CUDA;
    suf_stream = side->stream;
  }
  // suffix pass: each sequence's own keys, with the caller's masking (part sp)
  fa_status err_suf = FA_OK;
  if (err == FA_OK)
    err_suf = enqueue_paged(dev, q, k_pages, v_pages, page_table, cu_seqlens_q, kv_lens, num_seqs, total_q, max_q_len,
                            page_size, max_pages_per_seq, num_pages, Hq, Hkv, d, causal, scale, nullptr,
                            o_parts + part_rows * d * sp, lse_parts + part_rows * sp, scratch_suf, suf_bytes, 0,
                            suf_stream);
  // join even after an error, so that `stream` never runs ahead of work left on the side stream
  if (side && (cudaEventRecord(side->join, side->stream) != cudaSuccess ||
               cudaStreamWaitEvent(stream, side->join, 0) != cudaSuccess))
    return FA_ERR_CUDA;
  if (err != FA_OK) return err;
  if (err_suf != FA_OK) return err_suf;
  return fa::launch_merge(o_parts, lse_parts, sp + 1, total_q, Hq, d, o, nullptr, lse, false, stream) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status fa_merge_states(const float* o_parts, const float* lse_parts, int num_parts, int n_rows, int H, int d,
                          void* o, float* lse, fa_stream_t stream) {
  if (!o_parts || !lse_parts || !o) return FA_ERR_INVALID_ARG;
  if (num_parts <= 0 || n_rows <= 0 || H <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned16(o_parts) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FA_ERR_ALIGNMENT;
  fa_status err = FA_OK;
  if (!current_device(&err)) return err;
  return fa::launch_merge(o_parts, lse_parts, num_parts, n_rows, H, d, o, nullptr, lse, false, stream) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status fa_get_device_status(fa_stream_t stream, int* code, int* site) {
  if (!code) return FA_ERR_INVALID_ARG;
  fa_status err = FA_OK;
  const DeviceInfo* dev = current_device(&err);
  if (!dev) return err;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  DeviceStatus h{0, 0};
  if (cudaMemcpy(&h, dev->status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  const DeviceStatus zero{0, 0};
  if (cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  *code = (int)h.code;
  if (site) *site = (int)h.where;
  return FA_OK;
}

fa_status fa_selftest_wait_timeout(int limit_ms, int* code, int* site, fa_stream_t stream) {
  if (!code || limit_ms < 1 || limit_ms > 2000) return FA_ERR_INVALID_ARG;
  fa_status err = FA_OK;
  const DeviceInfo* dev = current_device(&err);
  if (!dev) return err;
  int dummy = 0;
  err = fa_get_device_status(stream, &dummy, nullptr);  // start from a clear status word
  if (err != FA_OK) return err;
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(dev->status, (uint64_t)limit_ms * 1000000ull);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  return fa_get_device_status(stream, code, site);
}

}  // extern "C"
