// Prints Philox4x32-10 outputs computed by PyTorch's header-only engine
// (ATen/core/PhiloxRNGEngine.h), an implementation independent of the oracle.
// Input lines on stdin: c0 c1 c2 c3 k0 k1 (decimal uint32); output: four words.
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdint>
#include <cstdio>

int main() {
  unsigned long long c0, c1, c2, c3, k0, k1;
  while (std::scanf("%llu %llu %llu %llu %llu %llu", &c0, &c1, &c2, &c3, &k0, &k1) == 6) {
    const uint64_t seed = (k1 << 32) | k0;
    const uint64_t subsequence = (c3 << 32) | c2;
    const uint64_t offset = (c1 << 32) | c0;
    at::philox_engine eng(seed, subsequence, offset);
    const uint32_t a = eng(), b = eng(), c = eng(), d = eng();
    std::printf("%u %u %u %u\n", a, b, c, d);
  }
  return 0;
}
