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
  float* part_o;    // [splits, T, H, 512] (decode split-K only)
  float* part_lse;  // [splits, T, H], base-2 log-sum-exp
  int* err;         // device error word
  KvSetDev set[2];
  int32_t nsets;
  int32_t total_tiles;
  int32_t T, H, num_seqs;
  int32_t groups;          // head groups per token
  int32_t heads_per_group;
  int32_t splits;          // CTAs per (token, group)
  int32_t tiles_per_split;
  float scale_log2;        // sm_scale * log2(e)
};

struct Plan {
  int groups;
  int heads_per_group;
  int nh;  // MMA N: 16, 32 or 64
  int splits;
  int tiles_per_split;
  int total_tiles;
  size_t part_o_bytes;
  size_t workspace_bytes;
};

// Launches the attention kernel (final outputs when args.splits == 1, partials otherwise)
// and, for splits > 1, the combine kernel. Returns cudaSuccess or the launch error.
cudaError_t launch_attention(const AttnArgs& args, const Plan& plan, cudaStream_t stream,
                             cudaEvent_t ev_start, cudaEvent_t ev_stop);

int* device_error_word();  // address of the device error word (host-side query helper)
cudaError_t read_and_clear_device_error(int* code);

}  // namespace smla
