// C-ABI layer of libsmla: argument validation with named diagnostics, the launch plan
// (head groups, split-K factor, workspace), the decode/prefill crossover table and the
// exported entry points declared in include/smla.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

// ------------------------------------------------------------------ diagnostics
struct Why {
  char* buf;
  size_t len;
  void set(const char* fmt, ...) {
    if (!buf || len == 0) return;
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, len, fmt, ap);
    va_end(ap);
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int row_bytes(int32_t format) { return format == SMLA_KV_BF16 ? kRowBf16 : kRowFp8; }

// Returns SMLA_OK, SMLA_ERR_INVALID or SMLA_ERR_UNSUPPORTED and names the field.
smla_status check_set(const smla_kv_set& s, const char* name, Why& why) {
  if (s.format != SMLA_KV_BF16 && s.format != SMLA_KV_FP8_E4M3_S128) {
    why.set("%s.format=%d unsupported: accepted 0 (SMLA_KV_BF16) or 1 (SMLA_KV_FP8_E4M3_S128)", name, s.format);
    return SMLA_ERR_UNSUPPORTED;
  }
  if (s.page_size != kPage) {
    why.set("%s.page_size=%d unsupported: accepted page_size is 64", name, s.page_size);
    return SMLA_ERR_UNSUPPORTED;
  }
  if (s.cache == nullptr || s.block_table == nullptr || s.seq_lens == nullptr || s.indices == nullptr) {
    why.set("%s: cache, block_table, seq_lens and indices must be non-NULL device pointers", name);
    return SMLA_ERR_INVALID;
  }
  if (!aligned16(s.cache)) {
    why.set("%s.cache must be 16-byte aligned", name);
    return SMLA_ERR_INVALID;
  }
  const int rb = row_bytes(s.format);
  if (s.row_stride_bytes < rb || (s.row_stride_bytes & 15) != 0) {
    why.set("%s.row_stride_bytes=%lld invalid: must be >= %d (row bytes of format %d) and a multiple of 16", name,
            static_cast<long long>(s.row_stride_bytes), rb, s.format);
    return SMLA_ERR_INVALID;
  }
  if (s.page_stride_bytes < kPage * s.row_stride_bytes || (s.page_stride_bytes & 15) != 0) {
    why.set("%s.page_stride_bytes=%lld invalid: must be >= 64*row_stride_bytes=%lld and a multiple of 16", name,
            static_cast<long long>(s.page_stride_bytes), static_cast<long long>(kPage * s.row_stride_bytes));
    return SMLA_ERR_INVALID;
  }
  if (s.num_pages < 1 || s.bt_stride < 1) {
    why.set("%s: num_pages=%d and bt_stride=%d must be >= 1", name, s.num_pages, s.bt_stride);
    return SMLA_ERR_INVALID;
  }
  if (s.num_pages > kMaxPages) {
    why.set("%s.num_pages=%d unsupported: at most %d pages (2^31 cache rows)", name, s.num_pages, kMaxPages);
    return SMLA_ERR_UNSUPPORTED;
  }
  if (s.topk < 1) {
    why.set("%s.topk=%d unsupported: accepted topk >= 1", name, s.topk);
    return SMLA_ERR_UNSUPPORTED;
  }
  if (s.idx_stride < s.topk) {
    why.set("%s.idx_stride=%lld invalid: must be >= topk=%d", name, static_cast<long long>(s.idx_stride), s.topk);
    return SMLA_ERR_INVALID;
  }
  return SMLA_OK;
}

smla_status check(const smla_params* p, Why& why) {
  if (p == nullptr) {
    why.set("params is NULL");
    return SMLA_ERR_INVALID;
  }
  if (p->d_qk != kDqk || p->d_v != kDv) {
    why.set("d_qk=%d d_v=%d unsupported: accepted family (d_qk, d_v) = (576, 512) (DSv4: 512 latent + 64 rope)",
            p->d_qk, p->d_v);
    return SMLA_ERR_UNSUPPORTED;
  }
  if (p->H < 1 || p->H > SMLA_MAX_HEADS) {
    why.set("H=%d unsupported: accepted num_heads 1..128 (any value, no padding)", p->H);
    return SMLA_ERR_UNSUPPORTED;
  }
  if (p->T < 0) {
    why.set("T=%d invalid: must be >= 0", p->T);
    return SMLA_ERR_INVALID;
  }
  if (p->num_seqs < 1) {
    why.set("num_seqs=%d invalid: must be >= 1", p->num_seqs);
    return SMLA_ERR_INVALID;
  }
  smla_status st = check_set(p->main, "main", why);
  if (st != SMLA_OK) return st;
  if (p->extra != nullptr) {
    st = check_set(*p->extra, "extra", why);
    if (st != SMLA_OK) return st;
  }
  if (p->q == nullptr || p->token_seq == nullptr || p->out == nullptr) {
    why.set("q, token_seq and out must be non-NULL device pointers");
    return SMLA_ERR_INVALID;
  }
  if (!aligned16(p->q) || (p->q_stride_t & 7) != 0 || (p->q_stride_h & 7) != 0 || p->q_stride_t < 0 ||
      p->q_stride_h < 0) {
    why.set("q must be 16-byte aligned with q_stride_t, q_stride_h non-negative multiples of 8 elements");
    return SMLA_ERR_INVALID;
  }
  if (!aligned16(p->out) || (p->out_stride_t & 7) != 0 || (p->out_stride_h & 7) != 0 || p->out_stride_h < kDv ||
      p->out_stride_t < 0) {
    why.set("out must be 16-byte aligned with out_stride_h >= 512 and out_stride_t, out_stride_h multiples of 8");
    return SMLA_ERR_INVALID;
  }
  if (p->lse != nullptr && p->lse_stride_t < p->H) {
    why.set("lse_stride_t=%lld invalid: must be >= H=%d", static_cast<long long>(p->lse_stride_t), p->H);
    return SMLA_ERR_INVALID;
  }
  if (!std::isfinite(p->sm_scale)) {
    why.set("sm_scale must be finite");
    return SMLA_ERR_INVALID;
  }
  return SMLA_OK;
}

// ------------------------------------------------------------------ device properties
int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

int ntiles_of(const smla_kv_set& s) { return (s.topk + kTile - 1) / kTile; }

// ------------------------------------------------------------------ plan
Plan make_plan(const smla_params* p, bool split_k) {
  Plan pl{};
  pl.groups = (p->H + kMaxGroupHeads - 1) / kMaxGroupHeads;
  const long long sms = sm_count();
  const int tiles_per_item = ntiles_of(p->main) + (p->extra ? ntiles_of(*p->extra) : 0);
  // a multiple of 8, so every group's first head starts a 16-byte run in the partial layout
  auto group_heads = [&](int g) { return (((p->H + g - 1) / g) + 7) & ~7; };
  // split-K with little work (small T): more, smaller head groups (up to four, at least 16
  // heads each, none empty) while the grid still fits one tile per SM, so more CTAs each carry
  // fewer heads on their latency-bound path (MMAs, softmax, epilogue); each row is then
  // gathered once per group, which at this size costs nothing measurable
  while (split_k && pl.groups < 4) {
    const int g2 = 2 * pl.groups;
    const int h2 = group_heads(g2);
    if (h2 < 16 || (g2 - 1) * h2 >= p->H || static_cast<long long>(p->T) * tiles_per_item * g2 > sms) break;
    pl.groups = g2;
  }
  pl.heads_per_group = group_heads(pl.groups);
  pl.nh = pl.heads_per_group <= 16 ? 16 : (pl.heads_per_group <= 32 ? 32 : 64);
  pl.tiles_per_item = tiles_per_item;
  pl.n_items = static_cast<long long>(p->T) * pl.groups;
  pl.total_tiles = pl.n_items * pl.tiles_per_item;
  pl.split = split_k ? 1 : 0;
  pl.max_slots = 1;
  if (pl.split) {
    // Contiguous flat tile ranges, one per persistent CTA; an item spans at most
    // ceil(tiles_per_item * nctas / total) + 1 ranges.
    pl.nctas = static_cast<int>(std::max<long long>(1, std::min(sms, pl.total_tiles)));
    const long long span = (static_cast<long long>(pl.tiles_per_item) * pl.nctas + pl.total_tiles - 1) /
                           std::max<long long>(1, pl.total_tiles);
    pl.max_slots = static_cast<int>(std::min<long long>(pl.nctas, span + 1));
  } else {
    pl.nctas = static_cast<int>(std::max<long long>(1, std::min(sms, pl.n_items)));
  }
  pl.part_o_bytes = 0;
  pl.workspace_bytes = 0;
  if (pl.split && p->T > 0) {
    const size_t n = static_cast<size_t>(pl.max_slots) * p->T * p->H;
    const size_t heads = static_cast<size_t>(pl.groups) * pl.heads_per_group;  // a multiple of 8
    pl.part_o_bytes = (static_cast<size_t>(pl.max_slots) * p->T * kDv * heads * sizeof(uint16_t) + 255) &
                      ~static_cast<size_t>(255);
    pl.workspace_bytes = pl.part_o_bytes + ((n * sizeof(float) + 255) & ~static_cast<size_t>(255));
  }
  return pl;
}

KvSetDev to_dev(const smla_kv_set& s) {
  KvSetDev d{};
  d.cache = static_cast<const uint8_t*>(s.cache);
  d.block_table = s.block_table;
  d.seq_lens = s.seq_lens;
  d.indices = s.indices;
  d.topk_length = s.topk_length;
  d.row_stride = s.row_stride_bytes;
  d.page_stride = s.page_stride_bytes;
  d.idx_stride = s.idx_stride;
  d.bt_stride = s.bt_stride;
  d.num_pages = s.num_pages;
  d.topk = s.topk;
  d.format = s.format;
  d.ntiles = ntiles_of(s);
  return d;
}

// ------------------------------------------------------------------ last CUDA error
thread_local char g_last_error[256] = {0};

// ------------------------------------------------------------------ timing hook
std::atomic<void*> g_ev_start{nullptr};
std::atomic<void*> g_ev_stop{nullptr};

smla_status run(const smla_params* p, cudaStream_t stream, bool split_k) {
  Why why{nullptr, 0};
  smla_status st = check(p, why);
  if (st != SMLA_OK) return st;
  if (p->T == 0) return SMLA_OK;
  const Plan pl = make_plan(p, split_k);
  if (pl.total_tiles >= (1ll << 31)) return SMLA_ERR_UNSUPPORTED;  // tile positions are 32-bit in the kernel
  if (pl.split) {
    if (p->workspace == nullptr || p->workspace_bytes < pl.workspace_bytes ||
        (reinterpret_cast<uintptr_t>(p->workspace) & 255u) != 0)
      return SMLA_ERR_WORKSPACE;
  }
  AttnArgs a{};
  a.q = static_cast<const uint16_t*>(p->q);
  a.q_stride_t = p->q_stride_t;
  a.q_stride_h = p->q_stride_h;
  a.token_seq = p->token_seq;
  a.sink = p->sink;
  a.out = static_cast<uint16_t*>(p->out);
  a.out_stride_t = p->out_stride_t;
  a.out_stride_h = p->out_stride_h;
  a.lse = p->lse;
  a.lse_stride_t = p->lse_stride_t;
  if (pl.split) {
    a.part_o = p->workspace;
    a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(p->workspace) + pl.part_o_bytes);
  }
  a.set[0] = to_dev(p->main);
  a.nsets = 1;
  if (p->extra) {
    a.set[1] = to_dev(*p->extra);
    a.nsets = 2;
  }
  a.tiles_per_item = pl.tiles_per_item;
  a.T = p->T;
  a.H = p->H;
  a.num_seqs = p->num_seqs;
  a.groups = pl.groups;
  a.heads_per_group = pl.heads_per_group;
  a.split = pl.split;
  a.nctas = pl.nctas;
  a.max_slots = pl.max_slots;
  a.nchunks = pl.groups * pl.heads_per_group / 8;
  a.n_items = pl.n_items;
  a.total_tiles = pl.total_tiles;
  a.scale_log2 = p->sm_scale * 1.4426950408889634f;
  const cudaError_t e = launch_attention(a, pl, stream, static_cast<cudaEvent_t>(g_ev_start.load()),
                                         static_cast<cudaEvent_t>(g_ev_stop.load()));
  return e == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

// ------------------------------------------------------------------ crossover table
struct CrossEntry {
  int32_t H, topk, format, max_tokens;
};
std::mutex g_cross_mu;
std::vector<CrossEntry> g_cross;

int32_t default_max_tokens(int32_t H) {
  // Without a calibration, use split-K while one CTA per (token, head group) would leave
  // more than half of the SMs idle.
  const int groups = (H + kMaxGroupHeads - 1) / kMaxGroupHeads;
  return std::max(1, sm_count() / (2 * groups));
}

}  // namespace

void note_cuda_error(cudaError_t e, const char* where) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

}  // namespace smla

using namespace smla;

extern "C" {

int smla_supported(const smla_params* p, char* why, size_t why_len) {
  Why w{why, why_len};
  if (why && why_len) why[0] = '\0';
  return check(p, w) == SMLA_OK ? 1 : 0;
}

size_t smla_workspace_size(const smla_params* p) {
  Why w{nullptr, 0};
  if (check(p, w) != SMLA_OK || p->T == 0) return 0;
  return make_plan(p, true).workspace_bytes;
}

smla_status smla_prefill(const smla_params* p, smla_stream_t stream) {
  return run(p, reinterpret_cast<cudaStream_t>(stream), false);
}

smla_status smla_decode(const smla_params* p, smla_stream_t stream) {
  return run(p, reinterpret_cast<cudaStream_t>(stream), true);
}

int32_t smla_decode_max_tokens(int32_t H, int32_t topk_total, int32_t format) {
  std::lock_guard<std::mutex> lk(g_cross_mu);
  const CrossEntry* best = nullptr;
  double best_d = 1e30;
  for (const auto& e : g_cross) {
    if (e.format != format) continue;
    const double d = std::fabs(std::log2(static_cast<double>(e.H)) - std::log2(static_cast<double>(std::max(1, H)))) +
                     std::fabs(std::log2(static_cast<double>(e.topk)) -
                               std::log2(static_cast<double>(std::max(1, topk_total))));
    if (d < best_d) {
      best_d = d;
      best = &e;
    }
  }
  return best ? best->max_tokens : default_max_tokens(H);
}

smla_status smla_forward(const smla_params* p, smla_stream_t stream) {
  Why w{nullptr, 0};
  const smla_status st = check(p, w);
  if (st != SMLA_OK) return st;
  const int32_t topk_total = p->main.topk + (p->extra ? p->extra->topk : 0);
  const bool decode = p->T <= smla_decode_max_tokens(p->H, topk_total, p->main.format);
  return run(p, reinterpret_cast<cudaStream_t>(stream), decode);
}

smla_status smla_set_crossover(const int32_t* entries, int32_t n) {
  if (n < 0 || (n > 0 && entries == nullptr)) return SMLA_ERR_INVALID;
  std::vector<CrossEntry> v;
  for (int32_t i = 0; i < n; ++i) {
    const CrossEntry e{entries[4 * i], entries[4 * i + 1], entries[4 * i + 2], entries[4 * i + 3]};
    if (e.H < 1 || e.H > SMLA_MAX_HEADS || e.topk < 1 || e.max_tokens < 0 || (e.format != 0 && e.format != 1))
      return SMLA_ERR_INVALID;
    v.push_back(e);
  }
  std::lock_guard<std::mutex> lk(g_cross_mu);
  g_cross.swap(v);
  return SMLA_OK;
}

smla_status smla_load_crossover(const char* json_path) {
  if (json_path == nullptr) return SMLA_ERR_INVALID;
  FILE* f = std::fopen(json_path, "rb");
  if (!f) return SMLA_ERR_INVALID;
  std::string text;
  char buf[4096];
  size_t n;
  while ((n = std::fread(buf, 1, sizeof(buf), f)) > 0) text.append(buf, n);
  std::fclose(f);
  const size_t vpos = text.find("\"version\"");
  const size_t epos = text.find("\"entries\"");
  if (vpos == std::string::npos || epos == std::string::npos) return SMLA_ERR_INVALID;
  const long version = std::strtol(text.c_str() + text.find(':', vpos) + 1, nullptr, 10);
  if (version != 1) {
    smla_set_crossover(nullptr, 0);
    return SMLA_ERR_UNSUPPORTED;
  }
  std::vector<int32_t> nums;
  const char* c = text.c_str() + text.find('[', epos);
  int depth = 0;
  for (; *c; ++c) {
    if (*c == '[') {
      ++depth;
    } else if (*c == ']') {
      if (--depth == 0) break;
    } else if (*c == '-' || (*c >= '0' && *c <= '9')) {
      char* end = nullptr;
      nums.push_back(static_cast<int32_t>(std::strtol(c, &end, 10)));
      c = end - 1;
    }
  }
  if (nums.size() % 4 != 0) return SMLA_ERR_INVALID;
  return smla_set_crossover(nums.data(), static_cast<int32_t>(nums.size() / 4));
}

const char* smla_status_string(smla_status s) {
  switch (s) {
    case SMLA_OK: return "SMLA_OK";
    case SMLA_ERR_INVALID: return "SMLA_ERR_INVALID: malformed arguments";
    case SMLA_ERR_UNSUPPORTED: return "SMLA_ERR_UNSUPPORTED: outside the supported envelope";
    case SMLA_ERR_WORKSPACE: return "SMLA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case SMLA_ERR_CUDA: return "SMLA_ERR_CUDA: CUDA runtime or launch failure";
    case SMLA_ERR_DEVICE: return "SMLA_ERR_DEVICE: a kernel gave up on a bounded wait";
  }
  return "unknown smla_status";
}

const char* smla_last_error(void) { return g_last_error; }

smla_status smla_device_error(int32_t* code) {
  if (code == nullptr) return SMLA_ERR_INVALID;
  int c = 0, cq = 0;
  cudaError_t e = read_and_clear_device_error(&c);
  if (e == cudaSuccess) e = read_and_clear_quant_error(&cq);
  if (e != cudaSuccess) {
    note_cuda_error(e, "reading the device error word");
    return SMLA_ERR_CUDA;
  }
  if (c == 0) c = cq;
  *code = c;
  return c == 0 ? SMLA_OK : SMLA_ERR_DEVICE;
}

smla_status smla_set_timing_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return SMLA_ERR_INVALID;
  g_ev_start.store(start_event);
  g_ev_stop.store(stop_event);
  return SMLA_OK;
}

size_t smla_struct_size(int32_t which) {
  return which == 0 ? sizeof(smla_params) : (which == 1 ? sizeof(smla_kv_set) : 0);
}

int32_t smla_version(void) { return (1 << 16) | 0; }

}  // extern "C"
