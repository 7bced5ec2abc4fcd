// SHA-256 as specified in FIPS 180-4.  The round constants and initial hash
// values are, by the standard's definition, the first 32 bits of the
// fractional parts of the cube roots of the first 64 primes and of the square
// roots of the first 8 primes; they are computed here exactly with integer
// roots rather than typed in.

#include "sha256.h"

#include <cstring>

namespace pa {

namespace {

using u128 = unsigned __int128;

// largest x with x^k <= n (k = 2 or 3), n < 2^110
uint64_t iroot(u128 n, int k) {
  uint64_t lo = 0, hi = 1ull << 40;
  while (lo < hi) {
    const uint64_t mid = lo + (hi - lo + 1) / 2;
    u128 p = 1;
    for (int i = 0; i < k; ++i) p *= mid;
    if (p <= n)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

struct Constants {
  uint32_t k[64];
  uint32_t h0[8];
  Constants() {
    int primes[64];
    int n = 0;
    for (int c = 2; n < 64; ++c) {
      bool prime = true;
      for (int d = 2; d * d <= c; ++d)
        if (c % d == 0) {
          prime = false;
          break;
        }
      if (prime) primes[n++] = c;
    }
    // frac(cbrt(p)) * 2^32 = cbrt(p * 2^96) mod 2^32, and likewise for sqrt
    for (int i = 0; i < 64; ++i)
      k[i] = static_cast<uint32_t>(iroot(static_cast<u128>(primes[i]) << 96, 3));
    for (int i = 0; i < 8; ++i)
      h0[i] = static_cast<uint32_t>(iroot(static_cast<u128>(primes[i]) << 64, 2));
  }
};

const Constants& consts() {
  static const Constants c;
  return c;
}

inline uint32_t rotr(uint32_t x, int r) { return (x >> r) | (x << (32 - r)); }

void compress(uint32_t h[8], const uint8_t block[64]) {
  const Constants& c = consts();
  uint32_t w[64];
  for (int t = 0; t < 16; ++t)
    w[t] = (uint32_t(block[4 * t]) << 24) | (uint32_t(block[4 * t + 1]) << 16) |
           (uint32_t(block[4 * t + 2]) << 8) | uint32_t(block[4 * t + 3]);
  for (int t = 16; t < 64; ++t) {
    const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
    const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
    w[t] = w[t - 16] + s0 + w[t - 7] + s1;
  }
  uint32_t a = h[0], b = h[1], cc = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
  for (int t = 0; t < 64; ++t) {
    const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
    const uint32_t ch = (e & f) ^ (~e & g);
    const uint32_t t1 = hh + S1 + ch + c.k[t] + w[t];
    const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
    const uint32_t maj = (a & b) ^ (a & cc) ^ (b & cc);
    const uint32_t t2 = S0 + maj;
    hh = g;
    g = f;
    f = e;
    e = d + t1;
    d = cc;
    cc = b;
    b = a;
    a = t1 + t2;
  }
  h[0] += a;
  h[1] += b;
  h[2] += cc;
  h[3] += d;
  h[4] += e;
  h[5] += f;
  h[6] += g;
  h[7] += hh;
}

}  // namespace

Sha256::Sha256() { std::memcpy(h, consts().h0, sizeof(h)); }

void Sha256::update(const void* data, size_t n) {
  const uint8_t* p = static_cast<const uint8_t*>(data);
  len += n;
  while (n > 0) {
    const size_t take = 64 - fill < n ? 64 - fill : n;
    std::memcpy(buf + fill, p, take);
    fill += take;
    p += take;
    n -= take;
    if (fill == 64) {
      compress(h, buf);
      fill = 0;
    }
  }
}

void Sha256::final(uint8_t out[32]) {
  const uint64_t bits = len * 8;
  const uint8_t one = 0x80, zero = 0;
  update(&one, 1);
  while (fill != 56) update(&zero, 1);
  uint8_t lenbuf[8];
  for (int i = 0; i < 8; ++i) lenbuf[i] = static_cast<uint8_t>(bits >> (56 - 8 * i));
  update(lenbuf, 8);
  for (int i = 0; i < 8; ++i) {
    out[4 * i] = static_cast<uint8_t>(h[i] >> 24);
    out[4 * i + 1] = static_cast<uint8_t>(h[i] >> 16);
    out[4 * i + 2] = static_cast<uint8_t>(h[i] >> 8);
    out[4 * i + 3] = static_cast<uint8_t>(h[i]);
  }
}

}  // namespace pa
