// Internal launch interface between the C-ABI layer (smla_api.cu) and the kernels
// (smla_kernels.cu). Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace smla {

constexpr int kDqk = 576;       // 512 latent + 64 rope channels
constexpr int kDv = 512;        // value = first 512 channels of the same row
constexpr int kPage = 64;       // tokens per cache page
constexpr int kTile = 128;      // gathered rows per tile = MMA M
constexpr int kRowBf16 = 1152;  // bytes of a bf16 row
constexpr int kRowFp8 = 656;    // bytes of an fp8 row: 512 e4m3 + 4 fp32 scales + 64 bf16 rope
constexpr int kMaxGroupHeads = 64;
constexpr int kMaxPages = 1 << 25;  // a cache row is addressed as (page << 6 | row) in 31 bits

struct KvSetDev {
  const uint8_t* cache;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* indices;
  const int32_t* topk_length;
  int64_t row_stride;
  int64_t page_stride;
  int64_t idx_stride;
  int32_t bt_stride;
  int32_t num_pages;
  int32_t topk;
  int32_t format;  // 0 bf16, 1 fp8
  int32_t ntiles;  // ceil(topk / kTile)
  int32_t pad_;
};

struct AttnArgs {
  const uint16_t* q;
  int64_t q_stride_t, q_stride_h;
  const int32_t* token_seq;
  const float* sink;
  uint16_t* out;
  int64_t out_stride_t, out_stride_h;
  float* lse;
  int64_t lse_stride_t;
  void* part_o;     // bf16 [max_slots, T, nchunks, 512, 8] normalised partial O^T in head chunks of 8
                    // (split schedule only)
  float* part_lse;  // [max_slots, T, H] base-2 log-sum-exp of each partial
  KvSetDev set[2];
  int32_t nsets;
  int32_t tiles_per_item;  // tiles of one (token, head group) item: main tiles then extra tiles
  int32_t T, H, num_seqs;
  int32_t groups;          // head groups per token
  int32_t heads_per_group;
  int32_t split;           // 0: whole items per CTA, final outputs; 1: contiguous tile ranges, partials
  int32_t nctas;           // persistent CTAs (grid size)
  int32_t max_slots;       // partial slots per item (split schedule)
  int32_t nchunks;         // head chunks of 8 per token in the partials: groups * heads_per_group / 8
  int64_t n_items;         // T * groups
  int64_t total_tiles;     // n_items * tiles_per_item
  float scale_log2;        // sm_scale * log2(e)
};

struct Plan {
  int groups;
  int heads_per_group;
  int nh;  // MMA N: 16, 32 or 64
  int split;
  int nctas;
  int max_slots;
  int tiles_per_item;
  long long n_items;
  long long total_tiles;
  size_t part_o_bytes;
  size_t workspace_bytes;
};

// First tile of CTA c in the split schedule: floor(c * total / nctas).
__host__ __device__ inline long long split_lo(long long c, long long total, long long nctas) {
  return c * total / nctas;
}
// The CTA whose split-schedule tile range contains flat tile x.
__host__ __device__ inline long long split_owner(long long x, long long total, long long nctas) {
  return ((x + 1) * nctas - 1) / total;
}

// Launches the persistent attention kernel (final outputs, or partials for the split
// schedule) and, for the split schedule, the combine kernel. Returns cudaSuccess or the
// launch error.
cudaError_t launch_attention(const AttnArgs& args, const Plan& plan, cudaStream_t stream,
                             cudaEvent_t ev_start, cudaEvent_t ev_stop);

cudaError_t read_and_clear_device_error(int* code);
// The cache writer's own device error word (its bounded waits), read and cleared.
cudaError_t read_and_clear_quant_error(int* code);

// Records a CUDA failure for smla_last_error (thread-local).
void note_cuda_error(cudaError_t e, const char* where);

}  // namespace smla
