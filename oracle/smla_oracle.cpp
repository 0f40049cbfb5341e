// Oracle for sparse top-k MLA attention — TEST INFRASTRUCTURE ONLY (see smla_oracle.h).
//
// Straight from the definition: gather the valid rows of the token's index set(s),
// dequantise each to fp64, then for every head form the scaled dot products, the
// sink-augmented softmax, the weighted sum of the value rows and the log-sum-exp.
// No blocking, no online rescaling, no fusion: one pass per (token, head).
#include "smla_oracle.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int kDqk = 576;   // 512 latent + 64 rope channels
constexpr int kDv = 512;    // value = first 512 channels of the same row
constexpr int kPage = 64;   // tokens per page

double bf16_value(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// OCP E4M3FN: sign, 4-bit exponent (bias 7), 3-bit mantissa; no infinities;
// exponent 1111 with mantissa 111 is NaN; exponent 0000 is subnormal (m/8 * 2^-6).
double e4m3_value(uint8_t code) {
  const int s = code >> 7;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  double v;
  if (e == 0xF && m == 0x7) {
    v = std::numeric_limits<double>::quiet_NaN();
  } else if (e == 0) {
    v = std::ldexp(static_cast<double>(m) / 8.0, -6);
  } else {
    v = std::ldexp(1.0 + static_cast<double>(m) / 8.0, e - 7);
  }
  return s ? -v : v;
}

// Dequantise one cache row into K[0..576).
void load_row(const oracle_kvset& s, const uint8_t* row, double* K) {
  if (s.fmt == 0) {
    for (int c = 0; c < kDqk; ++c) {
      uint16_t b;
      std::memcpy(&b, row + 2 * c, 2);
      K[c] = bf16_value(b);
    }
  } else {
    float scale[4];
    std::memcpy(scale, row + kDv, 16);
    for (int c = 0; c < kDv; ++c) K[c] = e4m3_value(row[c]) * static_cast<double>(scale[c / 128]);
    for (int c = 0; c < kDqk - kDv; ++c) {
      uint16_t b;
      std::memcpy(&b, row + kDv + 16 + 2 * c, 2);
      K[kDv + c] = bf16_value(b);
    }
  }
}

// Append the dequantised rows of every valid entry of token t in set s to rows.
void gather_set(const oracle_problem& p, const oracle_kvset& s, int t, std::vector<double>& rows) {
  const int seq = p.token_seq[t];
  if (seq < 0 || seq >= p.num_seqs) return;
  int width = s.topk;
  if (s.topk_length) width = std::min(width, std::max(0, s.topk_length[t]));
  const int32_t len = s.seq_lens[seq];
  for (int j = 0; j < width; ++j) {
    const int32_t i = s.indices[static_cast<int64_t>(t) * s.idx_stride + j];
    if (i < 0 || i >= len) continue;
    const int32_t lp = i / kPage;
    if (lp >= s.bt_stride) continue;
    const int32_t page = s.block_table[static_cast<int64_t>(seq) * s.bt_stride + lp];
    if (page < 0 || page >= s.num_pages) continue;
    const uint8_t* row = s.cache + static_cast<int64_t>(page) * s.page_stride +
                         static_cast<int64_t>(i % kPage) * s.row_stride;
    const size_t base = rows.size();
    rows.resize(base + kDqk);
    load_row(s, row, rows.data() + base);
  }
}

void one_token(const oracle_problem& p, int t, double* O, double* lse) {
  std::vector<double> rows;
  gather_set(p, p.main, t, rows);
  if (p.extra) gather_set(p, *p.extra, t, rows);
  const size_t n = rows.size() / kDqk;
  const double ninf = -std::numeric_limits<double>::infinity();
  std::vector<double> q(kDqk), x(n);
  for (int h = 0; h < p.H; ++h) {
    double* o = O + static_cast<int64_t>(h) * kDv;
    if (n == 0) {
      for (int c = 0; c < kDv; ++c) o[c] = 0.0;
      lse[h] = ninf;
      continue;
    }
    const uint16_t* qh = p.q + static_cast<int64_t>(t) * p.q_stride_t + static_cast<int64_t>(h) * p.q_stride_h;
    for (int c = 0; c < kDqk; ++c) q[c] = bf16_value(qh[c]);
    const double scale = static_cast<double>(p.sm_scale);
    for (size_t j = 0; j < n; ++j) {
      const double* K = rows.data() + j * kDqk;
      double acc = 0.0;
      for (int c = 0; c < kDqk; ++c) acc += q[c] * K[c];
      x[j] = scale * acc;
    }
    const bool has_sink = p.sink != nullptr;
    const double sigma = has_sink ? static_cast<double>(p.sink[h]) : ninf;
    double m = has_sink ? sigma : ninf;
    for (size_t j = 0; j < n; ++j) m = std::max(m, x[j]);
    double Z = 0.0;
    for (size_t j = 0; j < n; ++j) Z += std::exp(x[j] - m);
    const double D = has_sink ? Z + std::exp(sigma - m) : Z;
    for (int c = 0; c < kDv; ++c) o[c] = 0.0;
    for (size_t j = 0; j < n; ++j) {
      const double w = std::exp(x[j] - m) / D;
      const double* V = rows.data() + j * kDqk;
      for (int c = 0; c < kDv; ++c) o[c] += w * V[c];
    }
    lse[h] = m + std::log(Z);
  }
}

// ------------------------------------------------------------------ cache writer
// Packing new latent rows into the cache (the step the pages' benchmark runs before every
// measurement: flashinfer PR "add topk=256 prefill-dsv4 dispatch", conversation, the GB10
// benchmark's "Method" paragraph, where both sides' KV is packed by the same quantiser).
// The pages print no arithmetic for it; the reading taken here, per 128-channel latent block:
//   amax  = max |x_c|                            (exact)
//   scale = amax / 448 rounded to fp32            (1.0 when amax = 0); stored as fp32
//   y_c   = x_c / scale rounded to fp32           (the precision of the stored scale)
//   code  = the E4M3FN value nearest to y_c, ties to the even code, |y_c| > 448 -> 448
// and the 64 rope channels are rounded to bf16 (nearest, ties to even).

// bf16 bit pattern nearest to the fp32 value f (ties to the even pattern). The two
// candidates are the bf16 values that bracket f; the comparison is exact in fp64.
uint16_t bf16_nearest(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if (std::isnan(f)) return static_cast<uint16_t>((u >> 16) | 0x40);
  const uint32_t lo = u & 0xFFFF0000u;  // truncation toward zero
  const uint32_t hi = lo + 0x10000u;    // next bf16 away from zero
  float flo, fhi;
  std::memcpy(&flo, &lo, 4);
  std::memcpy(&fhi, &hi, 4);
  const double d_lo = std::fabs(static_cast<double>(f) - static_cast<double>(flo));
  const double d_hi = std::isinf(fhi) ? std::numeric_limits<double>::infinity()
                                      : std::fabs(static_cast<double>(fhi) - static_cast<double>(f));
  uint32_t pick;
  if (d_lo < d_hi) {
    pick = lo;
  } else if (d_hi < d_lo) {
    pick = hi;
  } else {
    pick = ((lo >> 16) & 1u) == 0 ? lo : hi;
  }
  // between the largest finite bf16 and 2^128 the halfway point decides overflow to infinity
  return static_cast<uint16_t>(pick >> 16);
}

// E4M3FN code nearest to y (saturating): searched over the 127 finite non-negative codes,
// whose values increase with the code.
uint8_t e4m3_nearest(float y) {
  static const std::vector<double> values = [] {
    std::vector<double> v(0x7F);
    for (int c = 0; c < 0x7F; ++c) v[c] = e4m3_value(static_cast<uint8_t>(c));
    return v;
  }();
  const uint8_t sign = std::signbit(y) ? 0x80 : 0x00;
  const double v = std::fabs(static_cast<double>(y));
  if (v >= 448.0) return sign | 0x7E;
  // c = largest code whose value is <= v
  const int c = static_cast<int>(std::upper_bound(values.begin(), values.end(), v) - values.begin()) - 1;
  if (values[c] == v) return sign | static_cast<uint8_t>(c);
  const double d_lo = v - values[c];
  const double d_hi = values[c + 1] - v;
  const int pick = d_lo < d_hi ? c : (d_hi < d_lo ? c + 1 : ((c & 1) == 0 ? c : c + 1));
  return sign | static_cast<uint8_t>(pick);
}

// One row of 576 fp32 values -> row bytes of format fmt.
void pack_row(const float* x, int32_t fmt, uint8_t* out) {
  if (fmt == 0) {
    for (int c = 0; c < kDqk; ++c) {
      const uint16_t b = bf16_nearest(x[c]);
      std::memcpy(out + 2 * c, &b, 2);
    }
    return;
  }
  for (int blk = 0; blk < 4; ++blk) {
    float amax = 0.0f;
    for (int c = 128 * blk; c < 128 * (blk + 1); ++c) amax = std::max(amax, std::fabs(x[c]));
    const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int c = 128 * blk; c < 128 * (blk + 1); ++c) {
      const float y = x[c] / scale;
      out[c] = e4m3_nearest(y);
    }
    std::memcpy(out + kDv + 4 * blk, &scale, 4);
  }
  for (int c = 0; c < kDqk - kDv; ++c) {
    const uint16_t b = bf16_nearest(x[kDv + c]);
    std::memcpy(out + kDv + 16 + 2 * c, &b, 2);
  }
}

bool malformed(const oracle_kvset& s) {
  return s.cache == nullptr || s.block_table == nullptr || s.seq_lens == nullptr ||
         s.indices == nullptr || s.topk < 0 || s.idx_stride < s.topk || (s.fmt != 0 && s.fmt != 1);
}

}  // namespace

extern "C" {

double oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }
double oracle_bf16_value(uint16_t bits) { return bf16_value(bits); }

int32_t oracle_threads(int32_t requested) {
  if (requested > 0) return requested;
  const unsigned hw = std::thread::hardware_concurrency();
  return hw ? static_cast<int32_t>(hw) : 1;
}

int oracle_pack_rows(const void* x, int32_t x_dtype, int64_t x_stride, int32_t n, int32_t fmt, uint8_t* out) {
  if (n < 0 || (n > 0 && (!x || !out)) || (fmt != 0 && fmt != 1) || (x_dtype != 0 && x_dtype != 1) ||
      x_stride < kDqk)
    return -1;
  const int row_bytes = fmt == 0 ? 2 * kDqk : kDv + 16 + 2 * (kDqk - kDv);
  // rows are independent: split them over threads
  const int32_t nt = std::max<int32_t>(1, std::min<int32_t>(oracle_threads(0), n / 1024 + 1));
  auto work = [&](int32_t r0, int32_t r1) {
    std::vector<float> row(kDqk);
    for (int32_t i = r0; i < r1; ++i) {
      for (int c = 0; c < kDqk; ++c) {
        if (x_dtype == 0) {
          uint16_t b;
          std::memcpy(&b, static_cast<const uint8_t*>(x) + 2 * (static_cast<int64_t>(i) * x_stride + c), 2);
          row[c] = static_cast<float>(bf16_value(b));
        } else {
          std::memcpy(&row[c], static_cast<const uint8_t*>(x) + 4 * (static_cast<int64_t>(i) * x_stride + c), 4);
        }
      }
      pack_row(row.data(), fmt, out + static_cast<int64_t>(i) * row_bytes);
    }
  };
  e4m3_nearest(0.0f);  // build the code table before the threads start
  std::vector<std::thread> pool;
  for (int32_t k = 1; k < nt; ++k)
    pool.emplace_back(work, static_cast<int32_t>(static_cast<int64_t>(n) * k / nt),
                      static_cast<int32_t>(static_cast<int64_t>(n) * (k + 1) / nt));
  work(0, static_cast<int32_t>(static_cast<int64_t>(n) / nt));
  for (auto& th : pool) th.join();
  return 0;
}

int oracle_attention(const oracle_problem* p, const int32_t* tokens, int32_t n, double* O,
                     double* lse, int32_t nthreads) {
  if (!p || !O || !lse || p->T < 0 || p->H < 1 || !p->q || !p->token_seq) return -1;
  if (malformed(p->main) || (p->extra && malformed(*p->extra))) return -1;
  const int32_t count = tokens ? n : p->T;
  if (count <= 0) return 0;
  const int32_t nt = std::min(oracle_threads(nthreads), count);
  std::atomic<int32_t> next{0};
  auto worker = [&]() {
    for (;;) {
      const int32_t k = next.fetch_add(1);
      if (k >= count) break;
      const int32_t t = tokens ? tokens[k] : k;
      one_token(*p, t, O + static_cast<int64_t>(k) * p->H * kDv, lse + static_cast<int64_t>(k) * p->H);
    }
  };
  std::vector<std::thread> pool;
  for (int32_t i = 1; i < nt; ++i) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  return 0;
}

}  // extern "C"
