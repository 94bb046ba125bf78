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

void make_buckets(const Spec& s, std::vector<Bucket>* out) {
  out->clear();
  auto push = [&](uint64_t lo, uint64_t hi) {
    Bucket b{};
    b.lo = lo;
    b.hi = hi;
    out->push_back(b);
  };
  if (s.bucket_bytes == 0) {
    push(0, s.N);
    return;
  }
  if (s.layers.empty()) {
    const uint64_t per = s.bucket_bytes / (uint64_t)s.esize;
    uint64_t hi = s.N;
    while (hi > 0) {
      const uint64_t lo = hi > per ? hi - per : 0;
      push(lo, hi);
      hi = lo;
    }
    return;
  }
  // tensors sit in forward order at increasing addresses; walk them backwards
  uint64_t top = s.N, cursor = s.N, bytes = 0;
  for (size_t i = s.layers.size(); i-- > 0;) {
    cursor -= s.layers[i];
    bytes += s.layers[i] * (uint64_t)s.esize;
    if (bytes >= s.bucket_bytes) {
      push(cursor, top);
      top = cursor;
      bytes = 0;
    }
  }
  if (top > 0) push(0, top);
}

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

  void add_segment(uint64_t lo, uint64_t len, const std::vector<int>& order, int inner, int groups) {
    if (len == 0) return;
    Segment g;
    g.order_off = (uint32_t)t->orders.size();
    g.inner = (uint16_t)inner;
    g.groups = (uint16_t)groups;
    for (int r : order) t->orders.push_back((uint8_t)r);
    const uint32_t seg = (uint32_t)t->segs.size();
    t->segs.push_back(g);
    const uint64_t tile = (uint64_t)s.tile_bytes / (uint64_t)s.esize;
    for (uint64_t a = lo, end = lo + len; a < end;) {
      const uint64_t next = std::min(end, (a / tile + 1) * tile);
      t->items.push_back(Item{a, (uint32_t)(next - a), seg});
      a = next;
    }
  }

  void fused_bucket(const Bucket& b) {
    const int P = s.P;
    const uint64_t n = b.hi - b.lo;
    std::vector<int> order(P);
    if (s.mode == kRankOrder) {
      std::iota(order.begin(), order.end(), 0);
      add_segment(b.lo, n, order, P, 1);
      return;
    }
    if (s.topo == kRing || s.topo == kMultiRing) {
      const int k = s.topo == kRing ? 1 : s.k;
      for (int j = 0; j < k; ++j) {
        const uint64_t slo = b.lo + part_lo(n, k, j), sn = part_len(n, k, j);
        const int m = s.topo == kRing ? 1 : mult[j];
        for (int c = 0; c < P; ++c) {
          for (int t2 = 0; t2 < P; ++t2) order[t2] = (int)((int64_t)((c + t2) % P) * m % P);
          add_segment(slo + part_lo(sn, P, c), part_len(sn, P, c), order, P, 1);
        }
      }
      return;
    }
    if (s.topo == kTorusND) {
      nd_segments(b.lo, n, 0, std::vector<int>(s.dims.size(), 0), order);
      return;
    }
    const int X = s.X, Y = s.Y;
    for (int c = 0; c < X; ++c) {
      const uint64_t clo = b.lo + part_lo(n, X, c), cn = part_len(n, X, c);
      for (int d = 0; d < Y; ++d) {
        for (int g = 0; g < Y; ++g)
          for (int h = 0; h < X; ++h) order[g * X + h] = ((d + g) % Y) * X + (c + h) % X;
        add_segment(clo + part_lo(cn, Y, d), part_len(cn, Y, d), order, X, Y);
      }
    }
  }

  // n-D torus: the range [lo, lo+n) is split along dim k into D_k chunks;
  // chunk tuple (c_0..c_{d-1}) folds, innermost first, the ranks with
  // coordinates x_k = (c_k + g_k) mod D_k for g_k = 0..D_k-1.
  void nd_segments(uint64_t lo, uint64_t n, int k, std::vector<int> ch, std::vector<int>& order) {
    const int d = (int)s.dims.size();
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
      add_segment(lo, n, order, s.dims[0], s.P / s.dims[0]);
      return;
    }
    for (int c = 0; c < s.dims[k]; ++c) {
      ch[k] = c;
      nd_segments(lo + part_lo(n, s.dims[k], c), part_len(n, s.dims[k], c), k + 1, ch, order);
    }
  }

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

uint32_t ldg_tile_bytes(uint64_t bytes_per_rank) {
  uint32_t t = kTileBytes;
  while (t > 1024 && bytes_per_rank < (uint64_t)t * 304) t >>= 1;
  return t;
}

uint32_t bulk_tile_bytes(int P) {
  uint32_t t = 16384;
  while (t > 256 && (uint64_t)t * (uint64_t)P > 65536) t >>= 1;
  return t;
}

bool ring_multipliers(int P, int k, std::vector<int>* out) {
  out->clear();
  if (P == 1) {
    out->push_back(1);
    return k == 1;
  }
  for (int c = 1; c < P && (int)out->size() < k; ++c)
    if (gcd_int(c, P) == 1) out->push_back(c);
  return (int)out->size() == k;
}

std::string validate(const Spec& s, bool* unsupported) {
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
    std::vector<int> m;
    if (s.k < 1) return "multi-ring needs k >= 1";
    if (!ring_multipliers(s.P, s.k, &m)) {
      *unsupported = true;
      return "multi-ring k exceeds the number of distinct rank orders t*s mod P (phi(P))";
    }
  } else if (s.topo == kTorus) {
    if (s.X < 1 || s.Y < 1 || (int64_t)s.X * s.Y != s.P) return "torus needs X * Y == P";
  } else if (s.topo == kTorusND) {
    if (s.dims.empty() || (int)s.dims.size() > kMaxDims) return "n-D torus needs 1..4 dims";
    int64_t prod = 1;
    for (int d : s.dims) {
      if (d < 1) return "n-D torus dims must be >= 1";
      prod *= d;
    }
    if (prod != s.P) return "n-D torus dims must multiply to P";
    if (s.dims.size() > 1 && s.dims.back() == 1) return "trailing dims of size 1 must be dropped";
  } else if (s.topo != kRing) {
    return "unknown topology kind";
  }
  if (s.bucket_bytes != 0 && s.bucket_bytes < (uint64_t)s.esize) return "bucket_bytes smaller than one element";
  if (!s.layers.empty()) {
    uint64_t sum = 0;
    for (uint64_t v : s.layers) {
      if (v == 0) return "a layer has zero elements";
      sum += v;
    }
    if (sum != s.N) return "layer sizes do not sum to N";
  }
  // work-item indices are 32-bit: up to 2^40 bytes per rank
  if (s.N * (uint64_t)s.esize > (1ull << 40)) {
    *unsupported = true;
    return "more than 2^40 bytes per rank";
  }
  return "";
}

bool build_tables(const Spec& s, bool with_steps, Tables* t) {
  try {
    *t = Tables();
    make_buckets(s, &t->buckets);
    Builder bld{s, t, with_steps, {}};
    if (s.topo == kMultiRing) ring_multipliers(s.P, s.k, &bld.mult);
    for (Bucket& b : t->buckets) {
      b.item_begin = (uint32_t)t->items.size();
      if (s.mode != kStepwise) bld.fused_bucket(b);
      b.item_end = (uint32_t)t->items.size();
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
    make_buckets(s, &t.buckets);
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
