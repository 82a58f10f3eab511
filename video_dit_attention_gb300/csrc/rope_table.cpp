// Host builders of the split-halves RoPE cos/sin tables (fp64 angles rounded to fp32).
//
// Difflet PR #153 (split RoPE commits): the rotary embedding pairs channel i of a head with
// channel i + D/2, and the pages build the cos/sin tables once per forward pass (permuted
// once instead of re-laid-out in every block); pad rows get the identity rotation. The
// Wan-style 3-D layout gives (t, h, w) 44/42/42 of the 128 channels with theta = 10000 per
// axis; tokens of the T x Hh x W latent grid are numbered row-major, t slowest.

#include <cmath>
#include <cstdint>

#include "../../include/dit_attn.h"

namespace {

void identity_rows(float* cos_out, float* sin_out, long long from, long long to, int half) {
  for (long long r = from; r < to; ++r)
    for (int i = 0; i < half; ++i) {
      cos_out[r * half + i] = 1.0f;
      sin_out[r * half + i] = 0.0f;
    }
}

}  // namespace

extern "C" int dit_rope_table_1d(float* cos_out, float* sin_out, int S_pad, int L, int D,
                                 double theta, int pos_offset) {
  if (!cos_out || !sin_out || S_pad < 0 || L < 0 || L > S_pad || !(theta > 0.0))
    return DIT_ERR_INVALID_ARG;
  if (D < 2 || (D % 2) != 0) return DIT_ERR_UNSUPPORTED;
  const int half = D / 2;
  for (int i = 0; i < half; ++i) {
    const double freq = std::pow(theta, -2.0 * i / D);
    for (int r = 0; r < L; ++r) {
      const double a = static_cast<double>(pos_offset + static_cast<long long>(r)) * freq;
      cos_out[static_cast<long long>(r) * half + i] = static_cast<float>(std::cos(a));
      sin_out[static_cast<long long>(r) * half + i] = static_cast<float>(std::sin(a));
    }
  }
  identity_rows(cos_out, sin_out, L, S_pad, half);
  return DIT_OK;
}

extern "C" int dit_rope_table_3d(float* cos_out, float* sin_out, int S_pad, int T, int Hh, int W,
                                 int D, int d_t, int d_h, int d_w, double theta) {
  if (!cos_out || !sin_out || S_pad < 0 || T < 0 || Hh < 0 || W < 0 || !(theta > 0.0))
    return DIT_ERR_INVALID_ARG;
  const long long n = static_cast<long long>(T) * Hh * W;
  if (n > S_pad) return DIT_ERR_INVALID_ARG;
  if (D < 2 || (D % 2) != 0 || d_t < 0 || d_h < 0 || d_w < 0 || (d_t % 2) || (d_h % 2) ||
      (d_w % 2) || d_t + d_h + d_w != D)
    return DIT_ERR_UNSUPPORTED;
  const int half = D / 2;
  const int widths[3] = {d_t, d_h, d_w};
  // freq[i] and axis[i] for every pair i: pairs [0, d_t/2) follow t, the next d_h/2 follow h,
  // the last d_w/2 follow w; within an axis block pair j has theta^(-2 j / d_axis).
  double freq[512];
  int axis[512];
  if (half > 512) return DIT_ERR_UNSUPPORTED;
  int i = 0;
  for (int a = 0; a < 3; ++a)
    for (int j = 0; j < widths[a] / 2; ++j, ++i) {
      freq[i] = std::pow(theta, -2.0 * j / widths[a]);
      axis[i] = a;
    }
  for (long long r = 0; r < n; ++r) {
    const long long coord[3] = {r / (static_cast<long long>(Hh) * W), (r / W) % Hh, r % W};
    for (int p = 0; p < half; ++p) {
      const double ang = static_cast<double>(coord[axis[p]]) * freq[p];
      cos_out[r * half + p] = static_cast<float>(std::cos(ang));
      sin_out[r * half + p] = static_cast<float>(std::sin(ang));
    }
  }
  identity_rows(cos_out, sin_out, n, S_pad, half);
  return DIT_OK;
}
