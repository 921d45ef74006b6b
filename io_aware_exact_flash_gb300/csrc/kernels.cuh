// Shared declarations between the C-ABI layer (api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include "ptx.cuh"

namespace fa {

// Tile shape of the tensor-core prefill kernel: each CTA owns two 128-row query tiles (one per
// softmax warpgroup) and streams 128-row key/value tiles.
constexpr int kBM = 128;   // query rows per tile (one TMEM lane per row)
constexpr int kBN = 128;   // keys per tile
constexpr int kQTiles = 2; // query tiles per CTA (ping-pong between the two softmax warpgroups)
constexpr int kPrefillThreads = 384;  // warps 0 (and 3, paged) TMA, warps 1-2 MMA, 4-11 softmax
// Registers per thread after the prefill CTA's split: warpgroup 0 (TMA, MMA, spare warps) drops
// to kRegsControl, the two softmax warpgroups rise to kRegsSoftmax. The sum stays within the
// 384 x 168 registers the CTA launches with (the launcher checks the compiled count).
constexpr int kRegsControl = 64;
constexpr int kRegsSoftmax = 216;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kPrefillThreads * 168, "register split too large");

struct alignas(64) PrefillParams {
  CUtensorMap tm_q;  // dense: (d, Hq, S, B)        paged: (d, Hq, total_q, 1)
  CUtensorMap tm_k;  // dense: (d, Hkv, S, B)       paged: (d, Hkv, page_size, num_pages)
  CUtensorMap tm_v;
  void* o;           // bf16 output (unused when o_f32 is set)
  float* o_f32;      // fp32 output instead of bf16 (a partial state for an LSE merge) or null
  float* lse;        // fp32 output or null
  int Hq, Hkv, group;
  int causal;
  float scale_log2;  // scale * log2(e)
  // dense
  int B, S;
  int kv_heads_per_chunk;  // unit order: kv heads whose query tiles are scheduled together
  int pair_units;          // dense causal: each CTA takes query-tile pairs i and T-1-i of one head
  // paged
  const int32_t* page_table;
  const int32_t* cu_seqlens_q;
  const int32_t* kv_lens;
  int page_size, max_pages_per_seq, num_pages, num_seqs;
  int pack;                // paged: query heads per tile row group (1, or the GQA group size:
                           // a tile row is then (token, head of the group), 128 / pack tokens)
  int kv_splits;           // paged: each unit's key tiles are split into this many contiguous
                           // ranges, each a unit of its own writing an fp32 partial state
  float* o_part;           // kv_splits > 1: fp32 [kv_splits, total_q, Hq, d] partial outputs
  float* lse_part;         // kv_splits > 1: fp32 [kv_splits, total_q, Hq] partial LSEs (natural log)
  int64_t total_q;         // rows of q/o/lse; no row at or past it is ever written
  const int2* work_list;   // (sequence, query-tile pair) items, heaviest first
  const int* work_count;
  DeviceStatus* status;
};

struct DecodeParams {
  const void* q;           // [total_q = num_seqs, Hq, d] bf16
  const void* k_pages;     // [num_pages, page_size, Hkv, d]
  const void* v_pages;
  const int32_t* page_table;
  const int32_t* cu_seqlens_q;
  const int32_t* kv_lens;
  void* o;                 // bf16 [total_q, Hq, d] (unused when o_f32 is set)
  float* o_f32;            // fp32 [total_q, Hq, d] instead of bf16, or null
  float* lse;              // fp32 [total_q, Hq] or null
  float* o_part;           // fp32 [num_splits, num_seqs, Hq, d]
  float* lse_part;         // fp32 [num_splits, num_seqs, Hq]  (log2 domain, scaled)
  int* counters;           // [num_seqs, Hkv / heads_per_cta] arrivals of the fused merge
  int num_seqs, Hq, Hkv, group, page_size, max_pages_per_seq, num_pages;
  int64_t total_q;
  int pages_per_split, num_splits;
  int heads_per_cta;       // kv heads one CTA handles
  float scale_log2;
  DeviceStatus* status;
};

// The CUDA-core decode kernel's grid has one y index per sequence, so a batch holds at most this
// many sequences on that kernel.
constexpr int kDecodeMaxSeqs = 65535;

// kv heads one decode CTA handles: the largest divisor of Hkv that is at most 8
inline int decode_heads_per_cta(int Hkv) {
  int h = Hkv <= 8 ? Hkv : 8;
  while (Hkv % h) --h;
  return h;
}

// Split-KV decode scratch: partial O | partial LSE | merge counters, each block 256-byte aligned.
inline size_t decode_scratch_bytes(int splits, int num_seqs, int Hq, int Hkv, int d) {
  if (splits <= 1) return 0;
  auto a = [](size_t x) { return (x + 255) / 256 * 256; };
  return a((size_t)splits * num_seqs * Hq * d * sizeof(float)) + a((size_t)splits * num_seqs * Hq * sizeof(float)) +
         a((size_t)num_seqs * (Hkv / decode_heads_per_cta(Hkv)) * sizeof(int));
}

inline void decode_scratch_layout(void* base, int splits, int num_seqs, int Hq, int d, DecodeParams& p) {
  auto a = [](size_t x) { return (x + 255) / 256 * 256; };
  char* c = static_cast<char*>(base);
  p.o_part = reinterpret_cast<float*>(c);
  c += a((size_t)splits * num_seqs * Hq * d * sizeof(float));
  p.lse_part = reinterpret_cast<float*>(c);
  c += a((size_t)splits * num_seqs * Hq * sizeof(float));
  p.counters = reinterpret_cast<int*>(c);
}

// Status word and SM count of the current device, for entry points defined outside api.cu.
// Returns 0 (FA_OK) or the fa_status code that describes why the device cannot be used.
int current_device_info(DeviceStatus** status, int* sm_count);

// Launchers (return cudaGetLastError() of the launch)
// Prefill launches have one CTA per work item, and a CTA that finishes takes over the items of CTAs
// that have not started; with the take-over off, paged work runs on a persistent grid instead
// (min(units, sm_count) CTAs looping over the units).
cudaError_t launch_prefill_dense(const PrefillParams& p, int d, int sm_count, cudaStream_t stream);
// after_plan (optional) is recorded on the stream between the planning kernel and the attention kernel.
cudaError_t launch_prefill_paged(const PrefillParams& p, int d, int sm_count, int max_items, int max_kv_tiles,
                                 int2* work_list, int* work_count, cudaStream_t stream,
                                 cudaEvent_t after_plan = nullptr);
cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t stream);
// The paged planning kernel alone: (sequence, tile pair) items longest first into work_list, their
// count into work_count[0], and work_count[1] = 0 (the unit counter of launch_decode_tc).
cudaError_t launch_plan_paged(const PrefillParams& p, int max_items, int max_kv_tiles, int2* work_list,
                              int* work_count, cudaStream_t stream);
// Decode / verify with the keys on the MMA's rows (decode_tc.cu): the query columns the softmax
// computes per unit (4, 8 or 16: the power of two >= max_q_len x group) for batches of at most
// max_rows (<= 16) query rows per (sequence, kv head) at d = 128, else 0.
int decode_tc_columns(int max_q_len, int group, int d, int max_rows);
// Plans the batch (p.pack must be 1 for the plan) and runs it on min(units, sm_count) persistent
// CTAs. p.tm_q's box is {64, group, 16 / group, 1}.
cudaError_t launch_decode_tc(const PrefillParams& p, int columns, int sm_count, int max_items, int max_kv_tiles,
                             int2* work_list, int* work_count, cudaStream_t stream, cudaEvent_t after_plan = nullptr);
// programmatic: launched as a programmatic dependent of the kernel before it on the stream (which
// should signal its dependents early); the merge waits for that kernel before reading.
cudaError_t launch_merge(const float* o_part, const float* lse_part, int num_parts, int n_rows, int H,
                         int d, void* o, float* o_f32, float* lse, bool log2_domain, cudaStream_t stream,
                         bool programmatic = false);

}  // namespace fa
