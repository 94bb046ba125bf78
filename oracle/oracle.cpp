/*
 * oracle.cpp -- TEST INFRASTRUCTURE ONLY (the oracle).
 *
 * A plain, slow, single-threaded CPU emulation of the synchronous-SGD gradient
 * all-reduce under its three schedules (ring, multi-ring, 2D-torus), plus an
 * independent per-element closed form of the same result.  Only the test
 * suite, the smoke check and the bench's CPU-baseline leg load this library.
 * It shares no code, header, table or helper with the CUDA library; the two
 * see the same inputs only through the seeded input generator module.
 *
 * Build: g++ -O2 -ffp-contract=off (no fast-math), so every float operation
 * below is one IEEE-754 binary32 operation rounded to nearest-even.
 *
 * Sources, cited by page title and section:
 *  [Ring]   Baidu ring-allreduce write-up, translated (final page of the
 *           Chinese translation), section "总结" (summary): gradients are
 *           averaged with the HPC ring all-reduce, a bandwidth-optimal
 *           algorithm (its reference 4, Patarasuk & Yuan 2009); the opening
 *           paragraphs: all-reduce works on one subset of the parameters at a
 *           time, output layers first, and every GPU sends and receives about
 *           twice the gradient size.
 *  [Multi]  "[论文解读] PowerAI DDL", abstract and section "提出的方法": a
 *           multi-ring communication pattern trading latency for bandwidth.
 *  [Torus]  "索尼发布新的方法，在ImageNet数据集上224秒内成功训练了ResNet-50"
 *           (Sony, ResNet-50 in 224 s), section "2D-Torus All-reduce",
 *           Fig. 1 and Fig. 2: GPUs on a logical 2D grid; the all-reduce is a
 *           horizontal reduce-scatter, a vertical all-reduce and a horizontal
 *           all-gather.
 *  [FP16]   same Sony page, section "训练设置" (training settings): gradient
 *           communication in half precision (FP16).
 *
 * Readings where the pages are silent (each is the plainest one; all are
 * listed in the design notes):
 *  R1 split of n elements into m parts: part i has n/m + (i < n%m) elements
 *     and starts at i*(n/m) + min(i, n%m).
 *  R2 buckets: bucket 0 holds the highest addresses (output layers); with a
 *     layer list, tensors are packed greedily in reverse forward order and a
 *     bucket closes once it holds >= bucket_bytes.
 *  R3 ring: position t sends to t+1; at reduce-scatter step s it sends chunk
 *     (t-s) mod m; the receiver adds; chunk c ends at position c-1, which
 *     applies the scale once; all-gather step s sends chunk (t+1-s) mod m.
 *  R4 multi-ring: slice j of k uses ring order pi_j(t) = t*s_j mod P, s_j the
 *     j-th smallest integer in [1, P) coprime to P (s_0 = 1 when P = 1).
 *  R5 torus: rank r = y*X + x; row rings pi(t) = y*X + t over X row chunks;
 *     row chunk c (owned at column c-1) runs a vertical ring pi(t) = t*X +
 *     (c-1 mod X) over its Y sub-chunks; then the horizontal all-gather.
 *  R6 fp16: every stored or sent value is binary16; each add is
 *     float(a) + float(b) in binary32; a result that is sent again is rounded
 *     to binary16 (RNE, subnormals kept, overflow to inf); the owner's last
 *     add stays binary32, is multiplied by the scale, then rounded once.
 *  R7 the scale is a binary32 multiplier applied once per element.
 *  R8 cost model: a worker has `links` network links; in a step every worker
 *     sends its messages at once, ring j's on link j mod links, so messages
 *     sharing a link queue behind each other; the step lasts alpha plus beta
 *     times the bytes of the busiest link.  One link per worker puts every
 *     schedule on the same hardware; links = k lets the k rings of a
 *     multi-ring run side by side.
 */
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <utility>
#include <vector>

namespace {

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16, written from the format definition (1 sign bit, 5     */
/* exponent bits with bias 15, 10 fraction bits; subnormals are             */
/* fraction * 2^-24; exponent field 31 encodes inf/NaN).                    */
/* ------------------------------------------------------------------------ */

uint32_t f32_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
float bits_f32(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

/* Exact widening: every binary16 value is a binary32 value. */
float half_to_float(uint16_t h) {
  const uint32_t sign = (uint32_t)(h >> 15) << 31;
  const uint32_t e = (h >> 10) & 0x1f;
  const uint32_t f = h & 0x3ff;
  if (e == 0) {
    /* zero or subnormal: f * 2^-24, exact in binary32 */
    float v = (float)f * bits_f32(0x33800000u); /* 2^-24 */
    return sign ? -v : v;
  }
  if (e == 31) return bits_f32(sign | 0x7f800000u | (f << 13)); /* inf / NaN */
  return bits_f32(sign | ((e - 15 + 127) << 23) | (f << 13));
}

/* Round-to-nearest, ties-to-even narrowing of a binary32 value.
 * |v| = M * 2^E with M the 24-bit integer significand.  The binary16 quantum
 * at magnitude 2^L is 2^(max(L,-14) - 10); round M * 2^E to a multiple of it. */
uint16_t float_to_half(float v) {
  const uint32_t u = f32_bits(v);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  const int e8 = (int)((u >> 23) & 0xff);
  const uint32_t frac = u & 0x7fffffu;
  if (e8 == 0xff) return frac ? (uint16_t)(sign | 0x7e00u) : (uint16_t)(sign | 0x7c00u);
  if (e8 == 0 && frac == 0) return sign;
  uint32_t M; int E;
  if (e8 == 0) { M = frac; E = -149; } else { M = frac | 0x800000u; E = e8 - 150; }
  int nbits = 0; for (uint32_t t = M; t; t >>= 1) ++nbits;
  const int L = E + nbits - 1;                 /* floor(log2 |v|) */
  int q = (L < -14 ? -14 : L) - 10;            /* exponent of the quantum */
  const int shift = q - E;                     /* >= 13 for every binary32 input */
  uint64_t m;
  if (shift >= 40) {
    m = 0;                                     /* below half the quantum */
  } else {
    const uint64_t MM = M;
    m = MM >> shift;
    const uint64_t rem = MM & ((1ull << shift) - 1);
    const uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (m & 1))) ++m;
  }
  if (m == 2048) { m = 1024; ++q; }            /* carried into the next binade */
  if (m < 1024) return (uint16_t)(sign | m);   /* subnormal (q == -24) or zero */
  const int e16 = q + 25;
  if (e16 >= 31) return (uint16_t)(sign | 0x7c00u); /* overflow to infinity */
  return (uint16_t)(sign | (e16 << 10) | (uint16_t)(m - 1024));
}

/* ------------------------------------------------------------------------ */
/* Configuration                                                            */
/* ------------------------------------------------------------------------ */

enum { DT_F32 = 0, DT_F16 = 1 };
enum { TOPO_RING = 0, TOPO_MULTIRING = 1, TOPO_TORUS = 2, TOPO_TORUS_ND = 3 };
constexpr int MAX_DIMS = 4;

struct Cfg {
  int P;
  uint64_t N;
  int dtype;
  int topo;
  int k;
  int X, Y;
  uint64_t bucket_bytes;
  std::vector<uint64_t> layers; /* numel per tensor, forward order; may be empty */
  std::vector<int> dims;        /* n-D torus: sizes of dims 0 (fastest) .. d-1 */
  uint64_t esize() const { return dtype == DT_F16 ? 2 : 4; }
};

/* R1 */
uint64_t part_size(uint64_t n, uint64_t m, uint64_t i) { return n / m + (i < n % m ? 1 : 0); }
uint64_t part_start(uint64_t n, uint64_t m, uint64_t i) { return i * (n / m) + std::min<uint64_t>(i, n % m); }
uint64_t part_of(uint64_t n, uint64_t m, uint64_t o) {
  const uint64_t base = n / m, rem = n % m, cut = rem * (base + 1);
  return o < cut ? o / (base + 1) : rem + (o - cut) / base;
}

int gcd(int a, int b) { while (b) { int t = a % b; a = b; b = t; } return a; }

/* R4: the multiplier of ring j. Returns false if fewer than k exist. */
bool ring_strides(int P, int k, std::vector<int>& s) {
  s.clear();
  if (P == 1) { s.push_back(1); return k == 1; }
  for (int c = 1; c < P && (int)s.size() < k; ++c)
    if (gcd(c, P) == 1) s.push_back(c);
  return (int)s.size() == k;
}

int validate(const Cfg& c) {
  if (c.P < 1 || c.N < 1) return -1;
  if (c.dtype != DT_F32 && c.dtype != DT_F16) return -2;
  if (c.topo == TOPO_MULTIRING) {
    std::vector<int> s;
    if (c.k < 1 || !ring_strides(c.P, c.k, s)) return -3;
  } else if (c.topo == TOPO_TORUS) {
    if (c.X < 1 || c.Y < 1 || (int64_t)c.X * c.Y != c.P) return -4;
  } else if (c.topo == TOPO_TORUS_ND) {
    if (c.dims.empty() || (int)c.dims.size() > MAX_DIMS) return -4;
    int64_t prod = 1;
    for (int d : c.dims) { if (d < 1) return -4; prod *= d; }
    if (prod != c.P) return -4;
  } else if (c.topo != TOPO_RING) {
    return -5;
  }
  if (!c.layers.empty()) {
    uint64_t s = 0;
    for (uint64_t n : c.layers) { if (n == 0) return -6; s += n; }
    if (s != c.N) return -6;
  }
  if (c.bucket_bytes && c.bucket_bytes < c.esize()) return -7;
  return 0;
}

/* R2: bucket b covers [first, second); index 0 = highest addresses. */
std::vector<std::pair<uint64_t, uint64_t>> make_buckets(const Cfg& c) {
  std::vector<std::pair<uint64_t, uint64_t>> b;
  if (c.bucket_bytes == 0) { b.push_back({0, c.N}); return b; }
  if (c.layers.empty()) {
    const uint64_t be = c.bucket_bytes / c.esize();
    for (uint64_t hi = c.N; hi > 0;) {
      const uint64_t lo = hi > be ? hi - be : 0;
      b.push_back({lo, hi});
      hi = lo;
    }
    return b;
  }
  /* tensors laid out in forward order at increasing addresses */
  uint64_t hi = c.N, lo = c.N, bytes = 0;
  for (size_t t = c.layers.size(); t-- > 0;) {
    lo -= c.layers[t];
    bytes += c.layers[t] * c.esize();
    if (bytes >= c.bucket_bytes) { b.push_back({lo, hi}); hi = lo; bytes = 0; }
  }
  if (hi > 0) b.push_back({0, hi});
  return b;
}

/* ------------------------------------------------------------------------ */
/* Rank buffers                                                             */
/* ------------------------------------------------------------------------ */

struct Bufs {
  void* const* p;
  int dtype;
  uint32_t raw(int r, uint64_t i) const {
    if (dtype == DT_F16) return ((const uint16_t*)p[r])[i];
    return f32_bits(((const float*)p[r])[i]);
  }
  void set_raw(int r, uint64_t i, uint32_t v) const {
    if (dtype == DT_F16) ((uint16_t*)p[r])[i] = (uint16_t)v;
    else ((float*)p[r])[i] = bits_f32(v);
  }
  float val(int r, uint64_t i) const { return raw_to_float(raw(r, i)); }
  float raw_to_float(uint32_t v) const { return dtype == DT_F16 ? half_to_float((uint16_t)v) : bits_f32(v); }
  /* store a binary32 result in the storage type (R6: binary16 RNE) */
  void put(int r, uint64_t i, float v) const {
    if (dtype == DT_F16) ((uint16_t*)p[r])[i] = float_to_half(v);
    else ((float*)p[r])[i] = v;
  }
};

/* One point-to-point message of one step. */
struct Msg {
  int src, dst;
  int ring;    /* which of the concurrent rings of the step carries it */
  uint64_t lo, hi;
  bool add;    /* reduce-scatter: receiver adds; all-gather: receiver copies */
  bool fin;    /* this add is the owner's last: scale, then store */
  std::vector<uint32_t> data;
};

struct Emu {
  const Cfg& c;
  const Bufs* b; /* null: count traffic only */
  float scale;
  int64_t stop_after; /* number of steps to run; < 0 = all */
  int links = 1;       /* network links per worker (cost model, R8) */
  uint64_t moved = 0, steps = 0;
  uint64_t step_load_sum = 0; /* sum over steps of the busiest link's elements (R8) */
  bool stopped = false;
  std::vector<Msg> pending;

  Emu(const Cfg& cfg, const Bufs* bufs, float s, int64_t stop) : c(cfg), b(bufs), scale(s), stop_after(stop) {}

  /* ring over positions ring[0..m-1] on elements [lo, hi); ring_id tells the
   * step's concurrent rings apart (multi-ring slice j) */
  void rs_send(const std::vector<int>& ring, uint64_t lo, uint64_t hi, int s, bool last_is_final,
               int ring_id = 0) {
    const int m = (int)ring.size();
    const uint64_t n = hi - lo;
    for (int t = 0; t < m; ++t) {
      const int ch = ((t - s) % m + m) % m;
      Msg g;
      g.src = ring[t];
      g.dst = ring[(t + 1) % m];
      g.ring = ring_id;
      g.lo = lo + part_start(n, m, ch);
      g.hi = g.lo + part_size(n, m, ch);
      g.add = true;
      g.fin = last_is_final && s == m - 2;
      pending.push_back(std::move(g));
    }
  }
  void ag_send(const std::vector<int>& ring, uint64_t lo, uint64_t hi, int s, int ring_id = 0) {
    const int m = (int)ring.size();
    const uint64_t n = hi - lo;
    for (int t = 0; t < m; ++t) {
      const int ch = ((t + 1 - s) % m + m) % m;
      Msg g;
      g.src = ring[t];
      g.dst = ring[(t + 1) % m];
      g.ring = ring_id;
      g.lo = lo + part_start(n, m, ch);
      g.hi = g.lo + part_size(n, m, ch);
      g.add = false;
      g.fin = false;
      pending.push_back(std::move(g));
    }
  }
  /* A ring of length one: its single member is the owner of everything. */
  void owner_scale_only(int r, uint64_t lo, uint64_t hi) {
    if (!b || stopped) return;
    for (uint64_t i = lo; i < hi; ++i) b->put(r, i, b->val(r, i) * scale);
  }

  /* Runs one step: every message of the step is read before any is applied,
   * so concurrent rings and in-place buffers cannot interfere. */
  void step() {
    if (stopped || (stop_after >= 0 && (int64_t)steps >= stop_after)) {
      stopped = true;
      pending.clear();
      return;
    }
    /* R8: the elements each (worker, link) pair sends in this step; ring j
     * uses link j mod links */
    std::vector<std::pair<std::pair<int, int>, uint64_t>> load;
    for (const Msg& g : pending) {
      const std::pair<int, int> key(g.src, g.ring % links);
      bool found = false;
      for (auto& e : load)
        if (e.first == key) { e.second += g.hi - g.lo; found = true; break; }
      if (!found) load.push_back({key, g.hi - g.lo});
    }
    uint64_t busiest = 0;
    for (const auto& e : load) busiest = std::max(busiest, e.second);
    for (Msg& g : pending) {
      moved += g.hi - g.lo;
      if (!b) continue;
      g.data.resize(g.hi - g.lo);
      for (uint64_t i = g.lo; i < g.hi; ++i) g.data[i - g.lo] = b->raw(g.src, i);
    }
    if (b) {
      for (const Msg& g : pending) {
        for (uint64_t i = g.lo; i < g.hi; ++i) {
          const uint32_t v = g.data[i - g.lo];
          if (!g.add) { b->set_raw(g.dst, i, v); continue; }
          const float sum = b->raw_to_float(v) + b->val(g.dst, i);
          if (g.fin) b->put(g.dst, i, sum * scale);
          else b->put(g.dst, i, sum);
        }
      }
    }
    pending.clear();
    ++steps;
    step_load_sum += busiest;
  }

  void ring_bucket(uint64_t lo, uint64_t hi) {
    std::vector<int> ring(c.P);
    for (int t = 0; t < c.P; ++t) ring[t] = t;
    for (int s = 0; s + 1 < c.P; ++s) { rs_send(ring, lo, hi, s, true); step(); }
    if (c.P == 1) owner_scale_only(0, lo, hi);
    for (int s = 0; s + 1 < c.P; ++s) { ag_send(ring, lo, hi, s); step(); }
  }

  void multiring_bucket(uint64_t lo, uint64_t hi) {
    std::vector<int> sj;
    ring_strides(c.P, c.k, sj);
    const uint64_t n = hi - lo;
    std::vector<std::vector<int>> rings(c.k, std::vector<int>(c.P));
    for (int j = 0; j < c.k; ++j)
      for (int t = 0; t < c.P; ++t) rings[j][t] = (int)(((int64_t)t * sj[j]) % c.P);
    for (int s = 0; s + 1 < c.P; ++s) {
      for (int j = 0; j < c.k; ++j) {
        const uint64_t a = lo + part_start(n, c.k, j);
        rs_send(rings[j], a, a + part_size(n, c.k, j), s, true, j);
      }
      step();
    }
    if (c.P == 1) owner_scale_only(0, lo, hi);
    for (int s = 0; s + 1 < c.P; ++s) {
      for (int j = 0; j < c.k; ++j) {
        const uint64_t a = lo + part_start(n, c.k, j);
        ag_send(rings[j], a, a + part_size(n, c.k, j), s, j);
      }
      step();
    }
  }

  void torus_bucket(uint64_t lo, uint64_t hi) {
    const int X = c.X, Y = c.Y;
    const uint64_t n = hi - lo;
    std::vector<std::vector<int>> rows(Y, std::vector<int>(X));
    for (int y = 0; y < Y; ++y)
      for (int t = 0; t < X; ++t) rows[y][t] = y * X + t;
    /* phase 1: horizontal reduce-scatter in every row; the row total is the
     * final value only when there is no vertical hop (Y == 1) */
    for (int s = 0; s + 1 < X; ++s) {
      for (int y = 0; y < Y; ++y) rs_send(rows[y], lo, hi, s, Y == 1);
      step();
    }
    if (X == 1 && Y == 1) owner_scale_only(0, lo, hi);
    /* phase 2: vertical all-reduce of row chunk c in column (c-1) mod X */
    std::vector<std::vector<int>> cols(X, std::vector<int>(Y));
    for (int ch = 0; ch < X; ++ch) {
      const int xc = ((ch - 1) % X + X) % X;
      for (int t = 0; t < Y; ++t) cols[ch][t] = t * X + xc;
    }
    for (int s = 0; s + 1 < Y; ++s) {
      for (int ch = 0; ch < X; ++ch) {
        const uint64_t a = lo + part_start(n, X, ch);
        rs_send(cols[ch], a, a + part_size(n, X, ch), s, true);
      }
      step();
    }
    for (int s = 0; s + 1 < Y; ++s) {
      for (int ch = 0; ch < X; ++ch) {
        const uint64_t a = lo + part_start(n, X, ch);
        ag_send(cols[ch], a, a + part_size(n, X, ch), s);
      }
      step();
    }
    /* phase 3: horizontal all-gather in every row */
    for (int s = 0; s + 1 < X; ++s) {
      for (int y = 0; y < Y; ++y) ag_send(rows[y], lo, hi, s);
      step();
    }
  }

  /* n-D torus, rank r = x0 + D0*(x1 + D1*(x2 + ...)).  Phase k < d-1:
   * reduce-scatter along dim k, every line of D_k ranks (other coordinates
   * fixed) on the range that line already reduced; the last dim all-reduces
   * its range (the owner's last add is final); then all-gathers along dims
   * d-2 .. 0.  The range a rank holds after the reduce-scatters along dims
   * 0..k-1 is: start from the bucket, take part (x_j + 1 mod D_j) of D_j
   * parts for j = 0..k-1 (its reduce-scatter ends at position c - 1). */
  void range_of(const std::vector<int>& x, int k, uint64_t lo, uint64_t hi, uint64_t* a, uint64_t* b) const {
    uint64_t s0 = lo, n = hi - lo;
    for (int j = 0; j < k; ++j) {
      const int D = c.dims[j];
      const uint64_t part = (uint64_t)((x[j] + 1) % D);
      s0 += part_start(n, D, part);
      n = part_size(n, D, part);
    }
    *a = s0;
    *b = s0 + n;
  }
  void coords(int r, std::vector<int>& x) const {
    x.assign(c.dims.size(), 0);
    for (size_t j = 0; j < c.dims.size(); ++j) { x[j] = r % c.dims[j]; r /= c.dims[j]; }
  }
  int rank_of(const std::vector<int>& x) const {
    int r = 0;
    for (size_t j = c.dims.size(); j-- > 0;) r = r * c.dims[j] + x[j];
    return r;
  }
  /* every line along dim k: the ranks in ring order (position = x_k) */
  std::vector<std::vector<int>> lines(int k) const {
    std::vector<std::vector<int>> out;
    std::vector<int> x;
    for (int r = 0; r < c.P; ++r) {
      coords(r, x);
      if (x[k] != 0) continue;
      std::vector<int> ring(c.dims[k]);
      for (int t = 0; t < c.dims[k]; ++t) { x[k] = t; ring[t] = rank_of(x); }
      out.push_back(ring);
    }
    return out;
  }
  void torus_nd_bucket(uint64_t lo, uint64_t hi) {
    const int d = (int)c.dims.size();
    std::vector<int> x;
    for (int k = 0; k < d; ++k) {
      const bool last_dim = (k == d - 1);
      const auto L = lines(k);
      for (int s = 0; s + 1 < c.dims[k]; ++s) {
        for (const auto& ring : L) {
          coords(ring[0], x);
          uint64_t a, b;
          range_of(x, k, lo, hi, &a, &b);
          rs_send(ring, a, b, s, last_dim);
        }
        step();
      }
      /* a ring of one at the last dim: the owner scales (only when P = 1,
       * since trailing dims of size 1 are dropped when the config is loaded) */
      if (last_dim && c.dims[k] == 1) owner_scale_only(0, lo, hi);
    }
    for (int k = d - 1; k >= 0; --k) {
      const auto L = lines(k);
      for (int s = 0; s + 1 < c.dims[k]; ++s) {
        for (const auto& ring : L) {
          coords(ring[0], x);
          uint64_t a, b;
          range_of(x, k, lo, hi, &a, &b);
          ag_send(ring, a, b, s);
        }
        step();
      }
    }
  }

  void run() {
    for (const auto& bk : make_buckets(c)) {
      if (c.topo == TOPO_RING) ring_bucket(bk.first, bk.second);
      else if (c.topo == TOPO_MULTIRING) multiring_bucket(bk.first, bk.second);
      else if (c.topo == TOPO_TORUS) torus_bucket(bk.first, bk.second);
      else torus_nd_bucket(bk.first, bk.second);
    }
  }
};

/* ------------------------------------------------------------------------ */
/* Closed form: the per-element result the schedule reaches.                */
/* out[i] = scale * Vfold_d( Hfold_c(row) for each row ), with the ring and */
/* the multi-ring as a single group of P.                                   */
/* ------------------------------------------------------------------------ */

struct Order { std::vector<int> rank; int inner, groups; std::vector<int> lev; /* n-D: level sizes */ };

Order fold_order(const Cfg& c, const std::vector<std::pair<uint64_t, uint64_t>>& bk, uint64_t i) {
  Order o;
  o.rank.resize(c.P);
  size_t b = 0;
  while (!(bk[b].first <= i && i < bk[b].second)) ++b;
  const uint64_t lo = bk[b].first, n = bk[b].second - bk[b].first, off = i - lo;
  if (c.topo == TOPO_RING) {
    const int ch = (int)part_of(n, c.P, off);
    for (int t = 0; t < c.P; ++t) o.rank[t] = (ch + t) % c.P;
    o.inner = c.P; o.groups = 1;
  } else if (c.topo == TOPO_MULTIRING) {
    std::vector<int> sj;
    ring_strides(c.P, c.k, sj);
    const int j = (int)part_of(n, c.k, off);
    const uint64_t a = part_start(n, c.k, j), nj = part_size(n, c.k, j);
    const int ch = (int)part_of(nj, c.P, off - a);
    for (int t = 0; t < c.P; ++t) o.rank[t] = (int)(((int64_t)((ch + t) % c.P) * sj[j]) % c.P);
    o.inner = c.P; o.groups = 1;
  } else if (c.topo == TOPO_TORUS) {
    const int ch = (int)part_of(n, c.X, off);
    const uint64_t a = part_start(n, c.X, ch), nc = part_size(n, c.X, ch);
    const int d = (int)part_of(nc, c.Y, off - a);
    for (int g = 0; g < c.Y; ++g)
      for (int h = 0; h < c.X; ++h) o.rank[g * c.X + h] = ((d + g) % c.Y) * c.X + (ch + h) % c.X;
    o.inner = c.X; o.groups = c.Y;
  } else {
    /* n-D torus: the chunk index along every dim, then the nested order:
     * position (g_0 + D0*(g_1 + D1*...)) holds the rank with coordinates
     * x_k = (c_k + g_k) mod D_k */
    const int d = (int)c.dims.size();
    std::vector<int> ch(d);
    uint64_t a = 0, m = n;
    for (int k = 0; k < d; ++k) {
      ch[k] = (int)part_of(m, c.dims[k], off - a);
      a += part_start(m, c.dims[k], ch[k]);
      m = part_size(m, c.dims[k], ch[k]);
    }
    for (int t = 0; t < c.P; ++t) {
      int rest = t, r = 0, stride = 1;
      for (int k = 0; k < d; ++k) {
        const int g = rest % c.dims[k];
        rest /= c.dims[k];
        r += ((ch[k] + g) % c.dims[k]) * stride;
        stride *= c.dims[k];
      }
      o.rank[t] = r;
    }
    o.lev = c.dims;
    o.inner = c.dims[0]; o.groups = c.P / c.dims[0];
  }
  return o;
}

float hop_add(float a, float b, bool last, int dtype);

/* Nested left fold: a group at level l is the left fold of its lev[l]
 * subgroups at level l-1 (level -1 = one rank's value).  Every add is rounded
 * to the storage type (R6) except the very last one, which is the add of the
 * last subgroup at the highest level of size > 1. */
float fold_group(const Order& o, const float* x, int l, int base, int top, int dtype) {
  if (l < 0) return x[o.rank[base]];
  int sub = 1;
  for (int j = 0; j < l; ++j) sub *= o.lev[j];
  float acc = fold_group(o, x, l - 1, base, top, dtype);
  for (int m = 1; m < o.lev[l]; ++m) {
    const float v = fold_group(o, x, l - 1, base + m * sub, top, dtype);
    const bool last = (l == top && m == o.lev[l] - 1);
    acc = hop_add(acc, v, last, dtype);
  }
  return acc;
}

/* R6: a result that travels again is rounded to the storage type. */
float hop_add(float a, float b, bool last, int dtype) {
  const float s = a + b;
  if (dtype == DT_F16 && !last) return half_to_float(float_to_half(s));
  return s;
}

/* x[r] = binary32 value of rank r's element; returns the stored result bits. */
uint32_t closed_form_value(const Cfg& c, const Order& o, const float* x, float scale) {
  if (!o.lev.empty()) {
    int top = -1;
    for (int l = 0; l < (int)o.lev.size(); ++l)
      if (o.lev[l] > 1) top = l;
    const float v = fold_group(o, x, (int)o.lev.size() - 1, 0, top, c.dtype);
    const float r = v * scale;
    return c.dtype == DT_F16 ? (uint32_t)float_to_half(r) : f32_bits(r);
  }
  float outer = 0.0f;
  for (int g = 0; g < o.groups; ++g) {
    float inner = x[o.rank[g * o.inner]];
    for (int h = 1; h < o.inner; ++h) {
      const bool last = (g == o.groups - 1) && (h == o.inner - 1) && o.groups == 1;
      inner = hop_add(inner, x[o.rank[g * o.inner + h]], last, c.dtype);
    }
    outer = (g == 0) ? inner : hop_add(outer, inner, g == o.groups - 1, c.dtype);
  }
  const float r = outer * scale;
  return c.dtype == DT_F16 ? (uint32_t)float_to_half(r) : f32_bits(r);
}

} /* namespace */

/* ======================================================================== */
/* C interface (ctypes)                                                      */
/* ======================================================================== */

extern "C" {

typedef struct {
  int32_t P;
  int32_t dtype;
  uint64_t N;
  int32_t topo;
  int32_t k;
  int32_t X;
  int32_t Y;
  uint64_t bucket_bytes;
  int64_t n_layers;
  const uint64_t* layers;
  int32_t ndims;     /* n-D torus (topo 3): number of dims, 1..4 */
  int32_t dims[4];   /* sizes, dim 0 varies fastest in the rank number */
} oracle_cfg;

static int load_cfg(const oracle_cfg* in, Cfg& c) {
  if (!in) return -100;
  c.P = in->P; c.N = in->N; c.dtype = in->dtype; c.topo = in->topo;
  c.k = in->k; c.X = in->X; c.Y = in->Y; c.bucket_bytes = in->bucket_bytes;
  c.layers.clear();
  if (in->n_layers > 0 && in->layers) c.layers.assign(in->layers, in->layers + in->n_layers);
  c.dims.clear();
  if (c.topo == TOPO_TORUS_ND) {
    if (in->ndims < 1 || in->ndims > MAX_DIMS) return -4;
    c.dims.assign(in->dims, in->dims + in->ndims);
    /* trailing dims of size 1 add no step; drop them so that the last
     * remaining dim carries the all-reduce with the final add */
    while (c.dims.size() > 1 && c.dims.back() == 1) c.dims.pop_back();
  }
  return validate(c);
}

/* Step-for-step emulation, in place on P host buffers of N elements each
 * (binary32, or binary16 bit patterns).  bufs == NULL counts traffic only.
 * stop_after >= 0 stops after that many communication steps (for traces).
 * Returns 0, or a negative code for an invalid configuration. */
int oracle_emulate(const oracle_cfg* cfg, void* const* bufs, float scale, int64_t stop_after,
                   uint64_t* elems_moved, uint64_t* steps) {
  Cfg c;
  const int rc = load_cfg(cfg, c);
  if (rc) return rc;
  Bufs b{bufs, c.dtype};
  Emu e(c, bufs ? &b : nullptr, scale, stop_after);
  e.run();
  if (elems_moved) *elems_moved = e.moved;
  if (steps) *steps = e.steps;
  return 0;
}

/* R8, alpha-beta time of the schedule on P real workers, each with `links`
 * network links: in every step all workers send at once; a worker's messages
 * of concurrent ring j travel on its link j mod links, one after another; the
 * step costs alpha + beta * (bytes on the busiest link of any worker); steps
 * add up.  From the emulation's own message lists. */
int oracle_cost(const oracle_cfg* cfg, double alpha, double beta, int32_t links, double* seconds) {
  Cfg c;
  const int rc = load_cfg(cfg, c);
  if (rc) return rc;
  if (links < 1) return -9;
  Emu e(c, nullptr, 1.0f, -1);
  e.links = links;
  e.run();
  *seconds = (double)e.steps * alpha + (double)e.step_load_sum * (double)c.esize() * beta;
  return 0;
}

/* The synchronous-SGD update that follows the all-reduce (Baidu write-up,
 * opening paragraph: each iteration runs forward, backward, the gradient
 * all-reduce, then the update; the pages' large-batch optimizer is LARS, whose
 * formula did not survive, so this is plain momentum SGD).  Per rank r and
 * element i, with g the all-reduced gradient as stored on rank r:
 *   d = g + wd * p;   v = mu * v + d;   p = p - lr * v
 * every product and sum rounded to binary32 separately (no fused multiply-add).
 * The all-reduce runs first, step by step (oracle_emulate); moms may be NULL
 * when mu == 0 (v is then d). */
int oracle_sgd(const oracle_cfg* cfg, void* const* grads, float* const* params, float* const* moms, float scale,
               float lr, float mu, float wd) {
  Cfg c;
  const int rc = load_cfg(cfg, c);
  if (rc) return rc;
  Bufs b{grads, c.dtype};
  Emu e(c, &b, scale, -1);
  e.run();
  for (int r = 0; r < c.P; ++r) {
    for (uint64_t i = 0; i < c.N; ++i) {
      const float g = b.val(r, i);
      float p = params[r][i];
      const float d = g + wd * p;
      float v = d;
      if (moms) {
        v = mu * moms[r][i] + d;
        moms[r][i] = v;
      }
      p = p - lr * v;
      params[r][i] = p;
    }
  }
  return 0;
}

/* Closed form at sampled elements.  x holds n_idx rows of P values: row s is
 * (rank 0 .. P-1) at element idx[s], in the storage type.  out receives the
 * n_idx results in the storage type. */
int oracle_closed_form(const oracle_cfg* cfg, const void* x, const uint64_t* idx, uint64_t n_idx,
                       float scale, void* out) {
  Cfg c;
  const int rc = load_cfg(cfg, c);
  if (rc) return rc;
  const auto bk = make_buckets(c);
  std::vector<float> row(c.P);
  for (uint64_t s = 0; s < n_idx; ++s) {
    if (idx[s] >= c.N) return -8;
    for (int r = 0; r < c.P; ++r) {
      if (c.dtype == DT_F16) row[r] = half_to_float(((const uint16_t*)x)[s * c.P + r]);
      else row[r] = ((const float*)x)[s * c.P + r];
    }
    const uint32_t v = closed_form_value(c, fold_order(c, bk, idx[s]), row.data(), scale);
    if (c.dtype == DT_F16) ((uint16_t*)out)[s] = (uint16_t)v;
    else ((float*)out)[s] = bits_f32(v);
  }
  return 0;
}

/* Fold order of element i: order_out[0..P-1] = ranks in the order they are
 * added; *inner = group length (X for the torus, P otherwise); *groups = Y or 1. */
int oracle_fold_order(const oracle_cfg* cfg, uint64_t i, int32_t* order_out, int32_t* inner, int32_t* groups) {
  Cfg c;
  const int rc = load_cfg(cfg, c);
  if (rc) return rc;
  if (i >= c.N) return -8;
  const Order o = fold_order(c, make_buckets(c), i);
  for (int t = 0; t < c.P; ++t) order_out[t] = o.rank[t];
  *inner = o.inner;
  *groups = o.groups;
  return 0;
}

/* Bucket table (R2). Returns the number of buckets (<= max written), or < 0. */
int64_t oracle_buckets(const oracle_cfg* cfg, uint64_t* begin, uint64_t* end, int64_t max) {
  Cfg c;
  const int rc = load_cfg(cfg, c);
  if (rc) return rc;
  const auto bk = make_buckets(c);
  for (int64_t b = 0; b < (int64_t)bk.size() && b < max; ++b) { begin[b] = bk[b].first; end[b] = bk[b].second; }
  return (int64_t)bk.size();
}

/* R4 ring multipliers; returns 0 or -3 when fewer than k distinct rings exist. */
int oracle_ring_strides(int32_t P, int32_t k, int32_t* out) {
  std::vector<int> s;
  if (P < 1 || k < 1 || !ring_strides(P, k, s)) return -3;
  for (int j = 0; j < k; ++j) out[j] = s[j];
  return 0;
}

/* fp64 reference of the plain mean: out[i] = scale * sum_r x_r[i], summed in
 * binary64 over the (already rounded) stored inputs, rank order. */
void oracle_ref64(int32_t P, uint64_t N, int32_t dtype, const void* const* bufs, double scale, double* out) {
  for (uint64_t i = 0; i < N; ++i) {
    double s = 0.0;
    for (int r = 0; r < P; ++r)
      s += dtype == DT_F16 ? (double)half_to_float(((const uint16_t*)bufs[r])[i]) : (double)((const float*)bufs[r])[i];
    out[i] = s * scale;
  }
}

void oracle_f32_to_f16(const float* in, uint16_t* out, uint64_t n) {
  for (uint64_t i = 0; i < n; ++i) out[i] = float_to_half(in[i]);
}

void oracle_f16_to_f32(const uint16_t* in, float* out, uint64_t n) {
  for (uint64_t i = 0; i < n; ++i) out[i] = half_to_float(in[i]);
}

/* Every binary32 bit pattern in [lo, hi) narrowed to binary16 (for the
 * exhaustive pin against an independent conversion). */
void oracle_f32_pattern_to_f16(uint64_t lo, uint64_t hi, uint16_t* out) {
  for (uint64_t p = lo; p < hi; ++p) out[p - lo] = float_to_half(bits_f32((uint32_t)p));
}

} /* extern "C" */
