// plan.cpp -- builds the tables that drive the all-reduce kernels.
//
// The schedules (sources by page title and section):
//  * ring: Baidu ring-allreduce write-up (final page), "总结" -- a chunked
//    reduce-scatter, then an all-gather, around a ring;
//  * multi-ring: "[论文解读] PowerAI DDL", abstract and "提出的方法" -- several
//    rings with different rank orders share the gradient;
//  * 2D-torus: "索尼发布新的方法，在ImageNet数据集上224秒内成功训练了ResNet-50",
//    "2D-Torus All-reduce", Fig. 1 / Fig. 2 -- horizontal reduce-scatter,
//    vertical all-reduce, horizontal all-gather;
//  * buckets in reverse-layer order: Baidu write-up, opening paragraphs.
//
// Fused mode turns each schedule into a per-element fold order: in a ring
// whose position t sends to t+1 and, at reduce-scatter step s, sends chunk
// (t - s) mod m, chunk c is first sent by position c and ends, fully reduced,
// at position c - 1; its value is the left fold of positions c, c+1, ...,
// c+m-1.  The torus nests two such folds: row chunk c is folded along each
// row from column c on, and its sub-chunk d is folded down the column from
// row d on.  Every element of one (bucket, slice, chunk) run shares one order,
// so the tables list runs ("segments") and tile-sized work items over them.
#include "plan.h"

#include <algorithm>
#include <new>
#include <numeric>

namespace ddl {
namespace {

// Split of n elements into m parts: part i has n/m + (i < n%m) elements and
// starts at i*(n/m) + min(i, n%m).
inline uint64_t part_len(uint64_t n, uint64_t m, uint64_t i) { return n / m + (i < n % m ? 1 : 0); }
inline uint64_t part_lo(uint64_t n, uint64_t m, uint64_t i) { return i * (n / m) + std::min(i, n % m); }

int gcd_int(int a, int b) {
  while (b) {
    const int r = a % b;
    a = b;
    b = r;
  }
  return a;
}

// The buckets of s from the highest addresses down: f(lo, hi) for each, in
// issue order; a false return stops the walk (and is returned).
template <typename F>
bool for_each_bucket(const Shape& s, F&& f) {
  if (s.bucket_bytes == 0) return f(uint64_t(0), s.N);
  if (s.n_layers == 0) {
    const uint64_t per = s.bucket_bytes / (uint64_t)s.esize;
    for (uint64_t hi = s.N; hi > 0;) {
      const uint64_t lo = hi > per ? hi - per : 0;
      if (!f(lo, hi)) return false;
      hi = lo;
    }
    return true;
  }
  // tensors sit in forward order at increasing addresses; walk them backwards
  uint64_t top = s.N, cursor = s.N, bytes = 0;
  for (uint64_t i = s.n_layers; i-- > 0;) {
    cursor -= s.layers[i];
    bytes += s.layers[i] * (uint64_t)s.esize;
    if (bytes >= s.bucket_bytes) {
      if (!f(cursor, top)) return false;
      top = cursor;
      bytes = 0;
    }
  }
  if (top > 0) return f(uint64_t(0), top);
  return true;
}

void make_buckets(const Shape& s, std::vector<Bucket>* out) {
  out->clear();
  for_each_bucket(s, [&](uint64_t lo, uint64_t hi) {
    Bucket b{};
    b.lo = lo;
    b.hi = hi;
    out->push_back(b);
    return true;
  });
}

// The fused tables of one plan shape, handed to a sink; fixed-size arrays
// only, so the allocation-free entry point can run it.
struct FusedWalk {
  const Shape& s;
  FusedSink* sink;
  int mult[kMaxP];
  int order[kMaxP];

  bool segment(uint64_t lo, uint64_t len, int inner, int groups) {
    if (len == 0) return true;
    if (!sink->segment(order, s.P, inner, groups)) return false;
    const uint64_t tile = (uint64_t)s.tile_bytes / (uint64_t)s.esize;
    for (uint64_t a = lo, end = lo + len; a < end;) {
      const uint64_t next = std::min(end, (a / tile + 1) * tile);
      if (!sink->item(a, (uint32_t)(next - a))) return false;
      a = next;
    }
    return true;
  }

  bool bucket(uint64_t lo, uint64_t hi) {
    const int P = s.P;
    const uint64_t n = hi - lo;
    if (s.mode == kRankOrder) {
      for (int t = 0; t < P; ++t) order[t] = t;
      return segment(lo, n, P, 1);
    }
    if (s.topo == kRing || s.topo == kMultiRing) {
      const int k = s.topo == kRing ? 1 : s.k;
      for (int j = 0; j < k; ++j) {
        const uint64_t slo = lo + part_lo(n, k, j), sn = part_len(n, k, j);
        const int m = s.topo == kRing ? 1 : mult[j];
        for (int c = 0; c < P; ++c) {
          for (int t = 0; t < P; ++t) order[t] = (int)((int64_t)((c + t) % P) * m % P);
          if (!segment(slo + part_lo(sn, P, c), part_len(sn, P, c), P, 1)) return false;
        }
      }
      return true;
    }
    if (s.topo == kTorusND) {
      int ch[kMaxDims] = {0, 0, 0, 0};
      return nd(lo, n, 0, ch);
    }
    const int X = s.X, Y = s.Y;
    for (int c = 0; c < X; ++c) {
      const uint64_t clo = lo + part_lo(n, X, c), cn = part_len(n, X, c);
      for (int d = 0; d < Y; ++d) {
        for (int g = 0; g < Y; ++g)
          for (int h = 0; h < X; ++h) order[g * X + h] = ((d + g) % Y) * X + (c + h) % X;
        if (!segment(clo + part_lo(cn, Y, d), part_len(cn, Y, d), X, Y)) return false;
      }
    }
    return true;
  }

  // n-D torus: the range [lo, lo+n) is split along dim k into D_k chunks;
  // chunk tuple (c_0..c_{d-1}) folds, innermost first, the ranks with
  // coordinates x_k = (c_k + g_k) mod D_k for g_k = 0..D_k-1.
  bool nd(uint64_t lo, uint64_t n, int k, int* ch) {
    const int d = s.ndims;
    if (k == d) {
      for (int t = 0; t < s.P; ++t) {
        int rest = t, r = 0, stride = 1;
        for (int j = 0; j < d; ++j) {
          const int g = rest % s.dims[j];
          rest /= s.dims[j];
          r += ((ch[j] + g) % s.dims[j]) * stride;
          stride *= s.dims[j];
        }
        order[t] = r;
      }
      return segment(lo, n, s.dims[0], s.P / s.dims[0]);
    }
    if (k >= kMaxDims) return false;  // check_shape keeps ndims <= kMaxDims
    for (int c = 0; c < s.dims[k]; ++c) {
      ch[k] = c;
      if (!nd(lo + part_lo(n, s.dims[k], c), part_len(n, s.dims[k], c), k + 1, ch)) return false;
    }
    return true;
  }
};

// The plan's tables, filled from the walk.
struct TableSink final : FusedSink {
  Tables* t;
  size_t b = 0;
  explicit TableSink(Tables* tab) : t(tab) {}
  bool bucket(uint64_t lo, uint64_t hi) override {
    if (b >= t->buckets.size() || t->buckets[b].lo != lo || t->buckets[b].hi != hi) return false;
    t->buckets[b].item_begin = (uint32_t)t->items.size();
    return true;
  }
  bool bucket_end() override {
    t->buckets[b++].item_end = (uint32_t)t->items.size();
    return true;
  }
  bool segment(const int* order, int P, int inner, int groups) override {
    Segment g;
    g.order_off = (uint32_t)t->orders.size();
    g.inner = (uint16_t)inner;
    g.groups = (uint16_t)groups;
    for (int r = 0; r < P; ++r) t->orders.push_back((uint8_t)order[r]);
    t->segs.push_back(g);
    return true;
  }
  bool item(uint64_t begin, uint32_t len) override {
    t->items.push_back(Item{begin, len, (uint32_t)(t->segs.size() - 1)});
    return true;
  }
};

// The step-by-step schedule: message lists (stepwise mode), traffic, steps
// and the cost model.
struct Builder {
  const Spec& s;
  Tables* t;
  bool with_steps;
  std::vector<int> mult;
  // cost model: links per worker; the elements each (worker, link) pair
  // sends in the step being built; their maximum summed over the steps
  int links = 1;
  std::vector<uint64_t> load;
  uint64_t busiest_sum = 0;

  // ---- message lists of the step-by-step schedule ----
  std::vector<Xfer> cur;

  // ring: which of the step's concurrent rings carries the message (the
  // multi-ring slice); it travels on link ring mod links of its sender
  void msg(uint64_t lo, uint64_t len, int src, int dst, uint32_t op, int ring = 0) {
    t->moved += (op == kScaleOnly) ? 0 : len;
    if (op != kScaleOnly) {
      const size_t at = (size_t)src * (size_t)links + (size_t)(ring % links);
      if (load.size() < (size_t)s.P * (size_t)links) load.assign((size_t)s.P * (size_t)links, 0);
      load[at] += len;
    }
    if (!with_steps) return;
    Xfer x{};
    x.lo = lo;
    x.len = len;
    x.src = (uint16_t)src;
    x.dst = (uint16_t)dst;
    x.op = op;
    cur.push_back(x);
  }
  // ring positions `ring`, elements [lo, lo+n), reduce-scatter step s
  void rs(const std::vector<int>& ring, uint64_t lo, uint64_t n, int step, bool owner_final, int ring_id = 0) {
    const int m = (int)ring.size();
    for (int p = 0; p < m; ++p) {
      const int c = ((p - step) % m + m) % m;
      const bool fin = owner_final && step == m - 2;
      msg(lo + part_lo(n, m, c), part_len(n, m, c), ring[p], ring[(p + 1) % m], fin ? kAddFinal : kAddHop,
          ring_id);
    }
  }
  void ag(const std::vector<int>& ring, uint64_t lo, uint64_t n, int step, int ring_id = 0) {
    const int m = (int)ring.size();
    for (int p = 0; p < m; ++p) {
      const int c = ((p + 1 - step) % m + m) % m;
      msg(lo + part_lo(n, m, c), part_len(n, m, c), ring[p], ring[(p + 1) % m], kCopy, ring_id);
    }
  }
  void close_step(bool communication) {
    if (communication) {
      ++t->nsteps;
      uint64_t busiest = 0;
      for (uint64_t v : load) busiest = std::max(busiest, v);
      busiest_sum += busiest;
    }
    std::fill(load.begin(), load.end(), 0);
    if (!with_steps) return;
    Step st{};
    st.xfer_begin = (uint32_t)t->xfers.size();
    uint64_t mx = 0;
    for (const Xfer& x : cur) {
      if (x.len == 0) continue;
      t->xfers.push_back(x);
      mx = std::max<uint64_t>(mx, x.len);
    }
    st.xfer_end = (uint32_t)t->xfers.size();
    st.max_len = mx;
    cur.clear();
    if (st.xfer_end > st.xfer_begin) t->steps.push_back(st);
  }

  void step_bucket(const Bucket& b) {
    const int P = s.P;
    const uint64_t n = b.hi - b.lo;
    if (P == 1) {  // a ring of one: the owner scales and nothing moves
      msg(b.lo, n, 0, 0, kScaleOnly);
      close_step(false);
      return;
    }
    if (s.topo == kRing || s.topo == kMultiRing) {
      const int k = s.topo == kRing ? 1 : s.k;
      std::vector<std::vector<int>> rings(k, std::vector<int>(P));
      for (int j = 0; j < k; ++j)
        for (int p = 0; p < P; ++p) rings[j][p] = (int)((int64_t)p * (s.topo == kRing ? 1 : mult[j]) % P);
      for (int st = 0; st < P - 1; ++st) {
        for (int j = 0; j < k; ++j) rs(rings[j], b.lo + part_lo(n, k, j), part_len(n, k, j), st, true, j);
        close_step(true);
      }
      for (int st = 0; st < P - 1; ++st) {
        for (int j = 0; j < k; ++j) ag(rings[j], b.lo + part_lo(n, k, j), part_len(n, k, j), st, j);
        close_step(true);
      }
      return;
    }
    if (s.topo == kTorusND) {
      nd_steps(b);
      return;
    }
    const int X = s.X, Y = s.Y;
    std::vector<std::vector<int>> row(Y, std::vector<int>(X)), col(X, std::vector<int>(Y));
    for (int y = 0; y < Y; ++y)
      for (int x = 0; x < X; ++x) row[y][x] = y * X + x;
    for (int c = 0; c < X; ++c)
      for (int y = 0; y < Y; ++y) col[c][y] = y * X + (c + X - 1) % X;  // row chunk c ends at column c-1
    for (int st = 0; st < X - 1; ++st) {
      for (int y = 0; y < Y; ++y) rs(row[y], b.lo, n, st, Y == 1);
      close_step(true);
    }
    for (int st = 0; st < Y - 1; ++st) {
      for (int c = 0; c < X; ++c) rs(col[c], b.lo + part_lo(n, X, c), part_len(n, X, c), st, true);
      close_step(true);
    }
    for (int st = 0; st < Y - 1; ++st) {
      for (int c = 0; c < X; ++c) ag(col[c], b.lo + part_lo(n, X, c), part_len(n, X, c), st);
      close_step(true);
    }
    for (int st = 0; st < X - 1; ++st) {
      for (int y = 0; y < Y; ++y) ag(row[y], b.lo, n, st);
      close_step(true);
    }
  }

  // n-D torus steps: reduce-scatter along dims 0..d-2 (each line of D_k ranks
  // on the range it has reduced so far), all-reduce along dim d-1, then
  // all-gather along dims d-2..0.  After the reduce-scatter along dim j a
  // rank at x_j holds part (x_j + 1) mod D_j of the range it started with.
  void nd_range(int r, int k, uint64_t lo, uint64_t n, uint64_t* a, uint64_t* m) const {
    uint64_t st = lo, len = n;
    for (int j = 0; j < k; ++j) {
      const int x = r % s.dims[j];
      r /= s.dims[j];
      const uint64_t part = (uint64_t)((x + 1) % s.dims[j]);
      st += part_lo(len, s.dims[j], part);
      len = part_len(len, s.dims[j], part);
    }
    *a = st;
    *m = len;
  }
  std::vector<std::vector<int>> nd_lines(int k) const {
    std::vector<std::vector<int>> out;
    int stride = 1;
    for (int j = 0; j < k; ++j) stride *= s.dims[j];
    for (int r = 0; r < s.P; ++r) {
      if ((r / stride) % s.dims[k] != 0) continue;
      std::vector<int> line(s.dims[k]);
      for (int t = 0; t < s.dims[k]; ++t) line[t] = r + t * stride;
      out.push_back(line);
    }
    return out;
  }
  void nd_steps(const Bucket& b) {
    const int d = (int)s.dims.size();
    const uint64_t n = b.hi - b.lo;
    for (int k = 0; k < d; ++k) {
      const auto lines = nd_lines(k);
      for (int st = 0; st < s.dims[k] - 1; ++st) {
        for (const auto& line : lines) {
          uint64_t a, m;
          nd_range(line[0], k, b.lo, n, &a, &m);
          rs(line, a, m, st, k == d - 1);
        }
        close_step(true);
      }
    }
    for (int k = d - 1; k >= 0; --k) {
      const auto lines = nd_lines(k);
      for (int st = 0; st < s.dims[k] - 1; ++st) {
        for (const auto& line : lines) {
          uint64_t a, m;
          nd_range(line[0], k, b.lo, n, &a, &m);
          ag(line, a, m, st);
        }
        close_step(true);
      }
    }
  }
};

}  // namespace

uint32_t ldg_tile_bytes(uint64_t bytes_per_rank, uint32_t floor) {
  uint32_t t = kTileBytes;
  while (t > floor && bytes_per_rank < (uint64_t)t * 304) t >>= 1;
  return t;
}

uint32_t fused_tile_floor(int P, int topo, int Y, int esize, int mode) {
  if (P >= kLatMinP) return 256;
  if (P >= kLatMinPHops && esize == 2 && mode == kFused && topo != kTorusND) return 256;
  const bool one_group = mode == kRankOrder || topo == kRing || topo == kMultiRing || (topo == kTorus && Y == 1);
  const bool unrounded = mode == kRankOrder || esize == 4;
  return one_group && unrounded ? 256 : 1024;
}

uint32_t bulk_tile_bytes(int P) {
  // at most kTileBytes: where a staged pass does not apply, the register pass
  // runs the same items, and its columns cover kTileBytes per rank
  uint32_t t = kTileBytes;
  while (t > 256 && (uint64_t)t * (uint64_t)P > 65536) t >>= 1;
  return t;
}

bool ring_multipliers_into(int P, int k, int* out) {
  if (P == 1) {
    out[0] = 1;
    return k == 1;
  }
  int found = 0;
  for (int c = 1; c < P && found < k; ++c)
    if (gcd_int(c, P) == 1) out[found++] = c;
  return found == k;
}

bool ring_multipliers(int P, int k, std::vector<int>* out) {
  out->clear();
  if (P < 1 || P > kMaxP || k < 1) return false;
  int m[kMaxP];
  const bool ok = ring_multipliers_into(P, k, m);
  const int n = P == 1 ? 1 : std::min(k, P - 1);
  out->assign(m, m + std::min(n, k));
  return ok;
}

Shape shape_of(const Spec& s) {
  Shape h;
  h.P = s.P;
  h.N = s.N;
  h.esize = s.esize;
  h.topo = s.topo;
  h.k = s.k;
  h.X = s.X;
  h.Y = s.Y;
  h.bucket_bytes = s.bucket_bytes;
  h.layers = s.layers.empty() ? nullptr : s.layers.data();
  h.n_layers = s.layers.size();
  h.mode = s.mode;
  h.tile_bytes = s.tile_bytes;
  h.ndims = (int)s.dims.size();
  for (int d = 0; d < kMaxDims && d < h.ndims; ++d) h.dims[d] = s.dims[d];
  return h;
}

const char* check_shape(const Shape& s, bool* unsupported) {
  *unsupported = false;
  if (s.P < 1) return "P must be >= 1";
  if (s.P > kMaxP) {
    *unsupported = true;
    return "P > 256 is not supported";
  }
  if (s.N < 1) return "N must be >= 1";
  if (s.esize != 4 && s.esize != 2) return "dtype must be DDL_FP32 or DDL_FP16";
  if (s.mode < kFused || s.mode > kRankOrder) return "unknown mode";
  if (s.topo == kMultiRing) {
    int m[kMaxP];
    if (s.k < 1) return "multi-ring needs k >= 1";
    if (!ring_multipliers_into(s.P, s.k, m)) {
      *unsupported = true;
      return "multi-ring k exceeds the number of distinct rank orders t*s mod P (phi(P))";
    }
  } else if (s.topo == kTorus) {
    if (s.X < 1 || s.Y < 1 || (int64_t)s.X * s.Y != s.P) return "torus needs X * Y == P";
  } else if (s.topo == kTorusND) {
    if (s.ndims < 1 || s.ndims > kMaxDims) return "n-D torus needs 1..4 dims";
    int64_t prod = 1;
    for (int d = 0; d < s.ndims; ++d) {
      if (s.dims[d] < 1) return "n-D torus dims must be >= 1";
      prod *= s.dims[d];
    }
    if (prod != s.P) return "n-D torus dims must multiply to P";
    if (s.ndims > 1 && s.dims[s.ndims - 1] == 1) return "trailing dims of size 1 must be dropped";
  } else if (s.topo != kRing) {
    return "unknown topology kind";
  }
  if (s.bucket_bytes != 0 && s.bucket_bytes < (uint64_t)s.esize) return "bucket_bytes smaller than one element";
  if (s.n_layers > 0) {
    if (!s.layers) return "layer list missing";
    uint64_t sum = 0;
    for (uint64_t i = 0; i < s.n_layers; ++i) {
      const uint64_t v = s.layers[i];
      if (v == 0) return "a layer has zero elements";
      if (v > s.N - sum) return "layer sizes exceed N";  // also keeps the sum from wrapping
      sum += v;
    }
    if (sum != s.N) return "layer sizes do not sum to N";
  }
  // work-item indices are 32-bit: up to 2^40 bytes per rank (compared
  // without forming N * esize, which could wrap)
  if (s.N > (1ull << 40) / (uint64_t)s.esize) {
    *unsupported = true;
    return "more than 2^40 bytes per rank";
  }
  if (s.tile_bytes < (uint32_t)s.esize || s.tile_bytes % (uint32_t)s.esize) return "bad tile size";
  return nullptr;
}

std::string validate(const Spec& s, bool* unsupported) {
  if ((size_t)s.dims.size() > (size_t)kMaxDims) {
    *unsupported = false;
    return "n-D torus needs 1..4 dims";
  }
  const char* why = check_shape(shape_of(s), unsupported);
  return why ? std::string(why) : std::string();
}

bool emit_fused(const Shape& s, FusedSink* sink) {
  FusedWalk walk{s, sink, {}, {}};
  if (s.topo == kMultiRing && !ring_multipliers_into(s.P, s.k, walk.mult)) return false;
  return for_each_bucket(s, [&](uint64_t lo, uint64_t hi) {
    return sink->bucket(lo, hi) && walk.bucket(lo, hi) && sink->bucket_end();
  });
}

bool build_tables(const Spec& s, bool with_steps, Tables* t) {
  try {
    *t = Tables();
    const Shape sh = shape_of(s);
    make_buckets(sh, &t->buckets);
    if (s.mode != kStepwise) {
      TableSink sink(t);
      if (!emit_fused(sh, &sink)) {
        *t = Tables();
        return false;
      }
    }
    Builder bld{s, t, with_steps, {}};
    if (s.topo == kMultiRing) ring_multipliers(s.P, s.k, &bld.mult);
    for (Bucket& b : t->buckets) {
      b.step_begin = (uint32_t)t->steps.size();
      bld.step_bucket(b);
      b.step_end = (uint32_t)t->steps.size();
    }
    // the kernels find segment s's rank order at s * P
    for (size_t i = 0; i < t->segs.size(); ++i)
      if (t->segs[i].order_off != (uint64_t)i * (uint64_t)s.P) return false;
    return true;
  } catch (const std::bad_alloc&) {
    *t = Tables();
    return false;
  }
}

bool schedule_cost(const Spec& s, double alpha, double beta, int links, double* seconds) {
  try {
    Tables t;
    make_buckets(shape_of(s), &t.buckets);
    Builder bld{s, &t, false, {}};
    // more links than concurrent rings carry nothing
    bld.links = std::max(1, std::min(links, s.topo == kMultiRing ? s.k : 1));
    if (s.topo == kMultiRing) ring_multipliers(s.P, s.k, &bld.mult);
    for (const Bucket& b : t.buckets) bld.step_bucket(b);
    *seconds = (double)t.nsteps * alpha + (double)bld.busiest_sum * (double)s.esize * beta;
    return true;
  } catch (const std::bad_alloc&) {
    return false;
  }
}

bool fold_order_of(const Spec& s, const Tables& t, uint64_t i, int32_t* order, int32_t* inner, int32_t* groups) {
  if (i >= s.N || s.mode == kStepwise) return false;
  // items are sorted by element within each bucket; buckets run downwards
  for (const Bucket& b : t.buckets) {
    if (i < b.lo || i >= b.hi) continue;
    auto first = t.items.begin() + b.item_begin, last = t.items.begin() + b.item_end;
    auto it = std::upper_bound(first, last, i, [](uint64_t v, const Item& x) { return v < x.begin; });
    if (it == first) return false;
    --it;
    if (i >= it->begin + it->len) return false;
    const Segment& g = t.segs[it->seg];
    for (int r = 0; r < s.P; ++r) order[r] = t.orders[g.order_off + r];
    *inner = g.inner;
    *groups = g.groups;
    return true;
  }
  return false;
}

}  // namespace ddl
