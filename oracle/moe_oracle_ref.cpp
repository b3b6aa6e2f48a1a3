// Plain C++ fp64 reference of one Mixture-of-Experts layer, forward and
// backward.  TEST INFRASTRUCTURE: only tests/ load it (through
// oracle/moe_oracle_ref.py).  It shares no code with the CUDA library nor
// with the numpy oracle beside it: it is a second, independent write-up of
// the same definitions, in loops, so that the two can be checked against
// each other.
//
// Definitions (UniEP page, "Unified Expert-Parallel MoE MegaKernel for LLM
// Training", section 1.1 and Figure 1; the SwiGLU expert is the MLP of the
// GraphPP page, sections 5.1-5.2; the token mapping is section 2.2,
// Algorithm 1, with one rank):
//   p[t] = softmax over all E of the fp32 logits (max-subtracted, fp64);
//   the k picks are the largest logits, ties to the lower expert index
//   (-0.0 == +0.0); w[t][j] = p of pick j, or that divided by the sum of the
//   picked p when renorm = 1;
//   the slots t*k+j are grouped by expert, stable in slot order;
//   per row: a = x W1_e^T, b = x W3_e^T, h = silu(a) * b, o = h W2_e^T;
//   y[t] = sum_j w[t][j] o[row(t, j)] + sum_s o[shared row s of t];
//   the backward of L = <dy, y>: dw = <dy, o>, dh = w dy W2_e,
//   dA = dh * b * s (1 + a (1 - s)), s = sigmoid(a), dB = dh * silu(a),
//   dx[t] = sum over the token's rows of dA W1_e + dB W3_e,
//   dW1_e = sum_rows dA^T x, dW3_e = sum_rows dB^T x, dW2_e = sum_rows (w dy)^T h,
//   and the router's Jacobian for dlogits.
// Inputs are the exact bits the GPU sees (bf16 as uint16, fp32 logits),
// widened to double; nothing is rounded on the way.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

double from_bf16(uint16_t v) {
  const uint32_t u = static_cast<uint32_t>(v) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

double sigmoid(double a) { return 1.0 / (1.0 + std::exp(-a)); }

}  // namespace

extern "C" {

// Router.  sel [T*k], w [T*k], p [T*E] (may be null).  Returns 0, or -1 if a
// logit is NaN or infinite.
int ref_route(const float* logits, int T, int E, int k, int renorm, int32_t* sel, double* w, double* p) {
  std::vector<double> z(E), ex(E);
  std::vector<char> taken(E);
  for (int t = 0; t < T; ++t) {
    double m = -INFINITY;
    for (int e = 0; e < E; ++e) {
      z[e] = logits[static_cast<size_t>(t) * E + e];
      if (!std::isfinite(z[e])) return -1;
      if (z[e] > m) m = z[e];
    }
    double s = 0.0;
    for (int e = 0; e < E; ++e) {
      ex[e] = std::exp(z[e] - m);
      s += ex[e];
    }
    if (p)
      for (int e = 0; e < E; ++e) p[static_cast<size_t>(t) * E + e] = ex[e] / s;
    for (int e = 0; e < E; ++e) taken[e] = 0;
    double psum = 0.0;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)  // strictly greater: the lower index wins a tie
        if (!taken[e] && (best < 0 || z[e] > z[best])) best = e;
      taken[best] = 1;
      sel[static_cast<size_t>(t) * k + j] = best;
      w[static_cast<size_t>(t) * k + j] = ex[best] / s;
      psum += ex[best] / s;
    }
    if (renorm)
      for (int j = 0; j < k; ++j) w[static_cast<size_t>(t) * k + j] /= psum;
  }
  return 0;
}

// Token mapping: a counting sort of the flat slots by expert, each expert's
// slots kept in flat-slot order.  counts [E], offsets [E+1], dest [T*k],
// row_token [T*k], row_slot [T*k].
int ref_permute(const int32_t* sel, int T, int E, int k, int32_t* counts, int32_t* offsets, int32_t* dest,
                int32_t* row_token, int32_t* row_slot) {
  const int R = T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int i = 0; i < R; ++i) {
    if (sel[i] < 0 || sel[i] >= E) return -1;
    ++counts[sel[i]];
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> next(offsets, offsets + E);
  for (int i = 0; i < R; ++i) {
    const int r = next[sel[i]]++;
    dest[i] = r;
    row_token[r] = i / k;
    row_slot[r] = i;
  }
  return 0;
}

// The layer's forward and backward.  x [T,d], dy [T,d], W1/W3 [E+S,f,d],
// W2 [E+S,d,f] as bf16 bits; logits [T,E] fp32.  Outputs (fp64, written in
// full): y [T,d], dx [T,d], dlogits [T,E], dW1/dW3 [E+S,f,d], dW2 [E+S,d,f],
// dw [T,k].  Returns 0, or -1 on a non-finite logit.
int ref_layer(const uint16_t* x, const float* logits, const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
              const uint16_t* dy, int T, int d, int f, int E, int k, int S, int renorm, double* y, double* dx,
              double* dlogits, double* dW1, double* dW3, double* dW2, double* dw) {
  const int R = T * k, Rs = R + S * T, nexp = E + S;
  std::vector<int32_t> sel(R), counts(E), offsets(E + 1), dest(R), row_token(R), row_slot(R);
  std::vector<double> w(R), p(static_cast<size_t>(T) * E);
  if (ref_route(logits, T, E, k, renorm, sel.data(), w.data(), p.data()) != 0) return -1;
  ref_permute(sel.data(), T, E, k, counts.data(), offsets.data(), dest.data(), row_token.data(), row_slot.data());

  std::vector<double> o(static_cast<size_t>(Rs) * d), dxp(static_cast<size_t>(Rs) * d), dwr(R, 0.0);
  for (size_t i = 0; i < static_cast<size_t>(nexp) * f * d; ++i) dW1[i] = dW3[i] = dW2[i] = 0.0;

  // One expert at a time owns its weight gradients; rows of one expert in
  // segment order.
#pragma omp parallel for schedule(dynamic, 1)
  for (int e = 0; e < nexp; ++e) {
    std::vector<double> xt(d), a(f), b(f), h(f), g(d), wg(d), dh(f), dA(f), dB(f);
    const uint16_t* W1e = W1 + static_cast<size_t>(e) * f * d;
    const uint16_t* W3e = W3 + static_cast<size_t>(e) * f * d;
    const uint16_t* W2e = W2 + static_cast<size_t>(e) * d * f;
    double* dW1e = dW1 + static_cast<size_t>(e) * f * d;
    double* dW3e = dW3 + static_cast<size_t>(e) * f * d;
    double* dW2e = dW2 + static_cast<size_t>(e) * d * f;
    const int r0 = e < E ? offsets[e] : R + (e - E) * T;
    const int r1 = e < E ? offsets[e + 1] : R + (e - E + 1) * T;
    for (int r = r0; r < r1; ++r) {
      const int t = e < E ? row_token[r] : r - r0;
      const double wr = e < E ? w[row_slot[r]] : 1.0;
      for (int i = 0; i < d; ++i) xt[i] = from_bf16(x[static_cast<size_t>(t) * d + i]);
      for (int j = 0; j < f; ++j) {
        double sa = 0.0, sb = 0.0;
        for (int i = 0; i < d; ++i) {
          sa += xt[i] * from_bf16(W1e[static_cast<size_t>(j) * d + i]);
          sb += xt[i] * from_bf16(W3e[static_cast<size_t>(j) * d + i]);
        }
        a[j] = sa;
        b[j] = sb;
        h[j] = sa * sigmoid(sa) * sb;
      }
      double* orow = o.data() + static_cast<size_t>(r) * d;
      for (int m = 0; m < d; ++m) {
        double s = 0.0;
        for (int j = 0; j < f; ++j) s += h[j] * from_bf16(W2e[static_cast<size_t>(m) * f + j]);
        orow[m] = s;
      }
      // backward of this row
      double dot = 0.0;
      for (int m = 0; m < d; ++m) {
        g[m] = from_bf16(dy[static_cast<size_t>(t) * d + m]);
        dot += g[m] * orow[m];
        wg[m] = wr * g[m];
      }
      if (e < E) dwr[r] = dot;
      for (int j = 0; j < f; ++j) {
        double s = 0.0;
        for (int m = 0; m < d; ++m) s += wg[m] * from_bf16(W2e[static_cast<size_t>(m) * f + j]);
        dh[j] = s;
        const double sg = sigmoid(a[j]);
        dA[j] = s * b[j] * sg * (1.0 + a[j] * (1.0 - sg));
        dB[j] = s * a[j] * sg;
      }
      double* xrow = dxp.data() + static_cast<size_t>(r) * d;
      for (int i = 0; i < d; ++i) {
        double s = 0.0;
        for (int j = 0; j < f; ++j)
          s += dA[j] * from_bf16(W1e[static_cast<size_t>(j) * d + i]) +
               dB[j] * from_bf16(W3e[static_cast<size_t>(j) * d + i]);
        xrow[i] = s;
      }
      for (int j = 0; j < f; ++j)
        for (int i = 0; i < d; ++i) {
          dW1e[static_cast<size_t>(j) * d + i] += dA[j] * xt[i];
          dW3e[static_cast<size_t>(j) * d + i] += dB[j] * xt[i];
        }
      for (int m = 0; m < d; ++m)
        for (int j = 0; j < f; ++j) dW2e[static_cast<size_t>(m) * f + j] += wg[m] * h[j];
    }
  }

  // Combine and the dx sum: the token's slots in order, then its shared rows.
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int i = 0; i < d; ++i) {
      double sy = 0.0, sx = 0.0;
      for (int j = 0; j < k; ++j) {
        const size_t r = static_cast<size_t>(dest[static_cast<size_t>(t) * k + j]);
        sy += w[static_cast<size_t>(t) * k + j] * o[r * d + i];
        sx += dxp[r * d + i];
      }
      for (int s = 0; s < S; ++s) {
        const size_t r = static_cast<size_t>(R) + static_cast<size_t>(s) * T + t;
        sy += o[r * d + i];
        sx += dxp[r * d + i];
      }
      y[static_cast<size_t>(t) * d + i] = sy;
      dx[static_cast<size_t>(t) * d + i] = sx;
    }
    // router: dL/dw, then the softmax Jacobian (renorm = 0) or that of the
    // softmax over the picked logits (renorm = 1)
    double inner = 0.0;
    for (int j = 0; j < k; ++j) {
      const size_t i = static_cast<size_t>(t) * k + j;
      dw[i] = dwr[dest[i]];
      inner += dw[i] * w[i];
    }
    for (int e = 0; e < E; ++e) {
      double picked_dw = 0.0, picked_w = 0.0;
      bool picked = false;
      for (int j = 0; j < k; ++j)
        if (sel[static_cast<size_t>(t) * k + j] == e) {
          picked = true;
          picked_dw = dw[static_cast<size_t>(t) * k + j];
          picked_w = w[static_cast<size_t>(t) * k + j];
        }
      double dz;
      if (renorm == 0)
        dz = p[static_cast<size_t>(t) * E + e] * ((picked ? picked_dw : 0.0) - inner);
      else
        dz = picked ? picked_w * (picked_dw - inner) : 0.0;
      dlogits[static_cast<size_t>(t) * E + e] = dz;
    }
  }
  return 0;
}

}  // extern "C"
