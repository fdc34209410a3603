// Reference ("oracle") implementation of one LAMB step on the CPU.
//
// TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
// benchmark's CPU-baseline leg; never by the product path.  It shares no code
// with the CUDA library.  The interface and the method are described in
// lamb_oracle.h; every step below follows the order given there:
//   LAMB (You et al., ICLR 2020, the layer-wise trust-ratio form of Adam) as
//   adopted by MegaScale (guided-reading digest, section 2: each layer's step
//   scaled by its own trust ratio, allowing 4x larger batches), applied to one rank's
//   ZeRO-2 shard (digest section 3, "Data parallelism (ZeRO-2 style)").
//
// Threads only split element ranges; every sum is formed per fixed block and
// the block sums are added in block order, so results do not depend on the
// number of threads.

#include "lamb_oracle.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int64_t kBlock = int64_t(1) << 16;  // elements per work block

template <class F>
void parallel_for(int64_t n, int threads, F&& f) {
  if (n <= 0) return;
  int64_t nt = std::min<int64_t>(threads, n);
  if (nt <= 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (;;) {
      int64_t i = next.fetch_add(1);
      if (i >= n) break;
      f(i);
    }
  };
  std::vector<std::thread> pool;
  pool.reserve(size_t(nt - 1));
  for (int64_t k = 1; k < nt; ++k) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
}

// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double decode_fp16(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int f = h & 0x3FF;
  double mag;
  if (e == 0) {
    mag = std::ldexp(double(f), -24);  // subnormal: f/1024 * 2^-14
  } else if (e == 31) {
    mag = f == 0 ? std::numeric_limits<double>::infinity()
                 : std::numeric_limits<double>::quiet_NaN();
  } else {
    mag = std::ldexp(1.0 + double(f) / 1024.0, e - 15);
  }
  return sign ? -mag : mag;
}

// bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
double decode_bf16(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 7) & 0xFF;
  const int f = h & 0x7F;
  double mag;
  if (e == 0) {
    mag = std::ldexp(double(f), -133);  // subnormal: f/128 * 2^-126
  } else if (e == 255) {
    mag = f == 0 ? std::numeric_limits<double>::infinity()
                 : std::numeric_limits<double>::quiet_NaN();
  } else {
    mag = std::ldexp(1.0 + double(f) / 128.0, e - 127);
  }
  return sign ? -mag : mag;
}

double decode(uint16_t bits, int32_t dtype) {
  return dtype == ORACLE_GRAD_FP16 ? decode_fp16(bits) : decode_bf16(bits);
}

// Keep the top 16 bits of the binary32 pattern, rounding the dropped 16 bits
// to nearest with ties to even; a carry out of the fraction correctly bumps
// the exponent (and overflows to infinity past the largest finite bf16).
uint16_t bf16_rne(float x) {
  uint32_t u;
  std::memcpy(&u, &x, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) {
    return uint16_t(((u >> 16) & 0x8000u) | 0x7FC0u);  // quiet NaN
  }
  uint32_t hi = u >> 16;
  const uint32_t lo = u & 0xFFFFu;
  if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1;
  return uint16_t(hi);
}

struct Block {
  int32_t tensor;
  int64_t begin, end;
};

void add_blocks(std::vector<Block>& out, int32_t i, int64_t n) {
  for (int64_t b = 0; b < n; b += kBlock) out.push_back({i, b, std::min(n, b + kBlock)});
}

struct Hyper {
  double b1, b2, eps, lr, bc1, bc2, gmul_c, S;
};

// Moments and direction for elements [b, e) of one tensor.  Stores m, v
// (rounded to fp32) and r (fp64) and returns the sums of w^2 and r^2.
void moments_and_direction(const Hyper& hp, double wd, const float* w, float* m, float* v,
                           const uint16_t* g, int32_t dtype, double* r, int64_t b, int64_t e,
                           double* sum_w2, double* sum_r2) {
  double sw = 0.0, sr = 0.0;
  for (int64_t j = b; j < e; ++j) {
    const double ghat = decode(g[j], dtype) / hp.S;       // unscale
    const double gp = hp.gmul_c * ghat;                     // clip
    const double mj = hp.b1 * double(m[j]) + (1.0 - hp.b1) * gp;
    const double vj = hp.b2 * double(v[j]) + (1.0 - hp.b2) * gp * gp;
    const double mhat = mj / hp.bc1;
    const double vhat = vj / hp.bc2;
    const double wj = double(w[j]);
    const double rj = mhat / (std::sqrt(vhat) + hp.eps) + wd * wj;
    sw += wj * wj;
    sr += rj * rj;
    m[j] = float(mj);
    v[j] = float(vj);
    r[j - b] = rj;
  }
  *sum_w2 = sw;
  *sum_r2 = sr;
}

double trust_ratio(double sum_w2, double sum_r2) {
  const double wn = std::sqrt(sum_w2);
  const double rn = std::sqrt(sum_r2);
  return (wn > 0.0 && rn > 0.0) ? wn / rn : 1.0;
}

void apply_update(double lr, double trust, float* w, uint16_t* w16, const double* r, int64_t b,
                  int64_t e) {
  for (int64_t j = b; j < e; ++j) {
    const float wn = float(double(w[j]) - lr * trust * r[j - b]);
    w[j] = wn;
    w16[j] = bf16_rne(wn);
  }
}

}  // namespace

extern "C" {

double oracle_decode_grad(uint16_t bits, int32_t grad_dtype) { return decode(bits, grad_dtype); }

uint16_t oracle_bf16_rne(float x) { return bf16_rne(x); }

void oracle_decode_grad_n(const uint16_t* bits, int64_t n, int32_t grad_dtype, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = decode(bits[i], grad_dtype);
}

void oracle_bf16_rne_n(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_rne(x[i]);
}

void oracle_loss_scale_update(float* scale, int32_t* good_steps, int32_t found_inf,
                              float growth, float backoff, int32_t growth_interval,
                              float min_scale, float max_scale) {
  float s = *scale;
  if (found_inf) {
    s = s * backoff;
    if (s < min_scale) s = min_scale;
    *good_steps = 0;
  } else {
    *good_steps += 1;
    if (*good_steps == growth_interval) {
      const float grown = s * growth;
      if (std::isfinite(grown)) s = grown > max_scale ? max_scale : grown;
      *good_steps = 0;
    }
  }
  *scale = s;
}

int oracle_lamb_step(int32_t n_tensors, const int64_t* sizes, const uint8_t* wd_flags,
                     float* const* w, float* const* m, float* const* v, uint16_t* const* w16,
                     const uint16_t* const* g, int32_t grad_dtype, double beta1, double beta2,
                     double eps, double weight_decay, double lr, int64_t t, double clip,
                     double loss_scale, const uint8_t* update_mask, int32_t n_threads,
                     int32_t* skipped, double* grad_norm, double* trust_out) {
  if (n_tensors < 0 || (n_tensors > 0 && (!sizes || !wd_flags || !g)) || !skipped ||
      !grad_norm || t < 1 || !(loss_scale > 0.0) || !std::isfinite(loss_scale) ||
      (grad_dtype != ORACLE_GRAD_BF16 && grad_dtype != ORACLE_GRAD_FP16)) {
    return -1;
  }
  for (int32_t i = 0; i < n_tensors; ++i) {
    if (sizes[i] < 0) return -1;
    if (sizes[i] > 0 && !g[i]) return -1;
    const bool upd = !update_mask || update_mask[i];
    if (upd && sizes[i] > 0 && (!w || !m || !v || !w16 || !w[i] || !m[i] || !v[i] || !w16[i]))
      return -1;
  }
  int threads = n_threads > 0 ? n_threads : int(std::thread::hardware_concurrency());
  if (threads < 1) threads = 1;

  // Unscale, finite check and global norm over every tensor of the shard.
  std::vector<Block> all;
  for (int32_t i = 0; i < n_tensors; ++i) add_blocks(all, i, sizes[i]);
  std::vector<double> part(all.size(), 0.0);
  std::vector<uint8_t> bad(all.size(), 0);
  parallel_for(int64_t(all.size()), threads, [&](int64_t k) {
    const Block& bl = all[size_t(k)];
    const uint16_t* gi = g[bl.tensor];
    double s = 0.0;
    uint8_t nf = 0;
    for (int64_t j = bl.begin; j < bl.end; ++j) {
      const double x = decode(gi[j], grad_dtype);
      if (!std::isfinite(x)) nf = 1;
      const double ghat = x / loss_scale;
      s += ghat * ghat;
    }
    part[size_t(k)] = s;
    bad[size_t(k)] = nf;
  });
  for (uint8_t b : bad) {
    if (b) {
      *skipped = 1;
      *grad_norm = std::numeric_limits<double>::infinity();
      return 0;
    }
  }
  double total = 0.0;
  for (double s : part) total += s;
  const double G = std::sqrt(total);
  *skipped = 0;
  *grad_norm = G;

  // Clip factor, then the bias corrections of step t.
  Hyper hp;
  hp.b1 = beta1;
  hp.b2 = beta2;
  hp.eps = eps;
  hp.lr = lr;
  hp.S = loss_scale;
  hp.gmul_c = (clip > 0.0 && G > clip) ? clip / G : 1.0;
  hp.bc1 = 1.0 - std::pow(beta1, double(t));
  hp.bc2 = 1.0 - std::pow(beta2, double(t));

  // Per tensor: moments, direction r, norms, trust ratio, update, bf16 copy.
  std::vector<int32_t> small, large;
  for (int32_t i = 0; i < n_tensors; ++i) {
    if (sizes[i] == 0 || (update_mask && !update_mask[i])) continue;
    (sizes[i] <= kBlock ? small : large).push_back(i);
  }

  parallel_for(int64_t(small.size()), threads, [&](int64_t k) {
    const int32_t i = small[size_t(k)];
    const int64_t n = sizes[i];
    const double wd = wd_flags[i] ? weight_decay : 0.0;
    std::vector<double> r(static_cast<size_t>(n));
    double sw, sr;
    moments_and_direction(hp, wd, w[i], m[i], v[i], g[i], grad_dtype, r.data(), 0, n, &sw, &sr);
    const double tr = trust_ratio(sw, sr);
    if (trust_out) trust_out[i] = tr;
    apply_update(lr, tr, w[i], w16[i], r.data(), 0, n);
  });

  for (int32_t i : large) {
    const int64_t n = sizes[i];
    const double wd = wd_flags[i] ? weight_decay : 0.0;
    std::vector<double> r(static_cast<size_t>(n));
    const int64_t nb = (n + kBlock - 1) / kBlock;
    std::vector<double> pw(static_cast<size_t>(nb)), pr(static_cast<size_t>(nb));
    parallel_for(nb, threads, [&](int64_t k) {
      const int64_t b = k * kBlock, e = std::min(n, b + kBlock);
      moments_and_direction(hp, wd, w[i], m[i], v[i], g[i], grad_dtype, r.data() + b, b, e,
                            &pw[size_t(k)], &pr[size_t(k)]);
    });
    double sw = 0.0, sr = 0.0;
    for (int64_t k = 0; k < nb; ++k) {
      sw += pw[size_t(k)];
      sr += pr[size_t(k)];
    }
    const double tr = trust_ratio(sw, sr);
    if (trust_out) trust_out[i] = tr;
    parallel_for(nb, threads, [&](int64_t k) {
      const int64_t b = k * kBlock, e = std::min(n, b + kBlock);
      apply_update(lr, tr, w[i], w16[i], r.data() + b, b, e);
    });
  }
  return 0;
}

}  // extern "C"
