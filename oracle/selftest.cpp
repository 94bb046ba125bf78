// selftest.cpp -- TEST INFRASTRUCTURE ONLY: drives the oracle's C interface on
// random problems, built together with oracle.cpp under AddressSanitizer and
// UndefinedBehaviorSanitizer by the test suite.  Checks that the step
// emulation equals the per-element closed form, that every rank ends with the
// same bits, and that 2(P-1)N elements moved; any memory or UB error aborts.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

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
  int32_t ndims;
  int32_t dims[4];
} oracle_cfg;
int oracle_emulate(const oracle_cfg*, void* const*, float, int64_t, uint64_t*, uint64_t*);
int oracle_closed_form(const oracle_cfg*, const void*, const uint64_t*, uint64_t, float, void*);
int oracle_ring_strides(int32_t, int32_t, int32_t*);
}

static uint64_t state = 0x243F6A8885A308D3ull;
static uint64_t next_u64() {  // xorshift64*
  state ^= state >> 12;
  state ^= state << 25;
  state ^= state >> 27;
  return state * 2685821657736338717ull;
}
static int uniform(int lo, int hi) { return lo + (int)(next_u64() % (uint64_t)(hi - lo + 1)); }

int main() {
  int failures = 0;
  for (int iter = 0; iter < 300; ++iter) {
    oracle_cfg c;
    std::memset(&c, 0, sizeof(c));
    c.P = uniform(1, 24);
    c.N = (uint64_t)uniform(1, 700);
    c.dtype = uniform(0, 1);
    c.topo = uniform(0, 3);
    if (c.topo == 1) {
      c.k = uniform(1, 3);
      std::vector<int32_t> s(c.k);
      if (oracle_ring_strides(c.P, c.k, s.data()) != 0) c.k = 1;
    } else if (c.topo == 2) {
      std::vector<int> d;
      for (int x = 1; x <= c.P; ++x)
        if (c.P % x == 0) d.push_back(x);
      c.X = d[uniform(0, (int)d.size() - 1)];
      c.Y = c.P / c.X;
    } else if (c.topo == 3) {
      int rest = c.P;
      c.ndims = uniform(1, 4);
      for (int j = 0; j < c.ndims - 1; ++j) {
        std::vector<int> d;
        for (int x = 1; x <= rest; ++x)
          if (rest % x == 0) d.push_back(x);
        c.dims[j] = d[uniform(0, (int)d.size() - 1)];
        rest /= c.dims[j];
      }
      c.dims[c.ndims - 1] = rest;
    }
    const uint64_t es = c.dtype ? 2 : 4;
    if (uniform(0, 2) == 0) c.bucket_bytes = (uint64_t)uniform((int)es, (int)(c.N * es));
    std::vector<std::vector<uint32_t>> raw(c.P, std::vector<uint32_t>(c.N));
    std::vector<std::vector<float>> f32(c.P, std::vector<float>(c.N));
    std::vector<std::vector<uint16_t>> f16(c.P, std::vector<uint16_t>(c.N));
    std::vector<void*> ptr(c.P);
    for (int r = 0; r < c.P; ++r) {
      for (uint64_t i = 0; i < c.N; ++i) {
        const double v = (double)((int64_t)(next_u64() % 2001) - 1000) * std::ldexp(1.0, uniform(-12, 4));
        f32[r][i] = (float)v;
        f16[r][i] = (uint16_t)(next_u64() & 0x7BFF);  // finite binary16 patterns
      }
      ptr[r] = c.dtype ? (void*)f16[r].data() : (void*)f32[r].data();
    }
    // inputs gathered per element before the in-place emulation
    std::vector<uint8_t> rows(c.N * c.P * es);
    for (uint64_t i = 0; i < c.N; ++i)
      for (int r = 0; r < c.P; ++r)
        std::memcpy(&rows[(i * c.P + r) * es], (const char*)ptr[r] + i * es, es);
    std::vector<uint64_t> idx(c.N);
    for (uint64_t i = 0; i < c.N; ++i) idx[i] = i;
    std::vector<uint8_t> closed(c.N * es);
    const float scale = 1.0f / (float)c.P;
    if (oracle_closed_form(&c, rows.data(), idx.data(), c.N, scale, closed.data()) != 0) {
      std::printf("config rejected at iter %d\n", iter);
      ++failures;
      continue;
    }
    uint64_t moved = 0, steps = 0;
    oracle_emulate(&c, ptr.data(), scale, -1, &moved, &steps);
    if (moved != 2ull * (uint64_t)(c.P - 1) * c.N) ++failures;
    for (int r = 0; r < c.P; ++r)
      if (std::memcmp(ptr[r], closed.data(), c.N * es) != 0) {
        std::printf("mismatch iter %d P=%d N=%llu topo=%d rank %d\n", iter, c.P, (unsigned long long)c.N, c.topo,
                    r);
        ++failures;
        break;
      }
  }
  std::printf("selftest failures: %d\n", failures);
  return failures ? 1 : 0;
}
