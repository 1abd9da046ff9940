// Host-side packing of 6-bit codes into bit-planes and of fp16 matrices into
// the stored page order.  The layout (documented in pw.h) puts, for every
// 16-row x 64-column chunk, the 32 weights that one GPU lane feeds to the
// tensor cores into one 32-bit word per plane.
#include <algorithm>
#include <cstring>
#include <thread>
#include <vector>

#include "pw.h"

namespace {

inline int word_in_tile(int kappa, int lane, int nk) {
  const int G = nk / 4, rem = nk % 4;
  const int gamma = kappa / 4, i = kappa % 4;
  return gamma < G ? gamma * 128 + lane * 4 + i : G * 128 + lane * rem + i;
}

}  // namespace

// Run fn(tile) for every 16-row tile, spread over the host's cores.
template <typename Fn>
void for_tiles(int ntiles, Fn fn) {
  const int hw = (int)std::max(1u, std::thread::hardware_concurrency());
  const int nth = std::min(hw, std::max(1, ntiles / 8));
  if (nth <= 1) {
    for (int t = 0; t < ntiles; ++t) fn(t);
    return;
  }
  std::vector<std::thread> th;
  for (int i = 0; i < nth; ++i)
    th.emplace_back([=] {
      for (int t = i; t < ntiles; t += nth) fn(t);
    });
  for (auto& x : th) x.join();
}

extern "C" pw_status pw_pack_planes(const uint8_t* code6, int R, int C, uint32_t* const planes_out[6]) {
  if (!code6 || !planes_out || R <= 0 || C <= 0 || R % 16 || C % 64) return PW_ERR_INVALID_ARG;
  for (int p = 0; p < 6; ++p)
    if (!planes_out[p]) return PW_ERR_INVALID_ARG;
  const int nk = C / 64;
  uint32_t* outs[6];
  for (int p = 0; p < 6; ++p) outs[p] = planes_out[p];
  for_tiles(R / 16, [=](int tau) {
    for (int kappa = 0; kappa < nk; ++kappa) {
      for (int lane = 0; lane < 32; ++lane) {
        const int g = lane >> 2, t = lane & 3;
        uint32_t word[6] = {0, 0, 0, 0, 0, 0};
        // gather the lane's 32 weights: k picks (row half, column half), h the
        // even/odd column of a pair, s the 16-column step
        for (int k = 0; k < 4; ++k) {
          const int row = 16 * tau + g + 8 * (k >> 1);
          for (int h = 0; h < 2; ++h) {
            for (int s = 0; s < 4; ++s) {
              const int col = 64 * kappa + 16 * s + 2 * t + 8 * (k & 1) + h;
              const uint32_t code = code6[(size_t)row * C + col] & 63u;
              const int q = 8 * k + 4 * h + s;
              for (int p = 0; p < 6; ++p) word[p] |= ((code >> (5 - p)) & 1u) << ((q + 5 - p) & 31);
            }
          }
        }
        const size_t wi = (size_t)tau * nk * 32 + word_in_tile(kappa, lane, nk);
        for (int p = 0; p < 6; ++p) outs[p][wi] = word[p];
      }
    }
  });
  return PW_OK;
}

extern "C" pw_status pw_pack_f16(const uint16_t* w, int R, int C, uint16_t* out) {
  if (!w || !out || R <= 0 || C <= 0 || R % 16 || C % 64) return PW_ERR_INVALID_ARG;
  const int nk = C / 64;
  for_tiles(R / 16, [=](int tau) {
    size_t o = (size_t)tau * 16 * C;
    for (int kappa = 0; kappa < nk; ++kappa)
      for (int s = 0; s < 4; ++s)
        for (int lane = 0; lane < 32; ++lane) {
          const int g = lane >> 2, t = lane & 3;
          for (int a = 0; a < 4; ++a) {
            const int row = 16 * tau + g + 8 * (a & 1);
            for (int h = 0; h < 2; ++h) {
              const int col = 64 * kappa + 16 * s + 2 * t + 8 * (a >> 1) + h;
              out[o++] = w[(size_t)row * C + col];
            }
          }
        }
  });
  return PW_OK;
}
