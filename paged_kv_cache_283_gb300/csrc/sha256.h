// SHA-256 (FIPS 180-4), used to name prefix-cache blocks.  Host only.
#pragma once

#include <cstddef>
#include <cstdint>

namespace pa {

struct Sha256 {
  uint32_t h[8];
  uint8_t buf[64];
  uint64_t len = 0;  // bytes absorbed
  size_t fill = 0;   // bytes waiting in buf

  Sha256();
  void update(const void* data, size_t n);
  void final(uint8_t out[32]);
};

}  // namespace pa
