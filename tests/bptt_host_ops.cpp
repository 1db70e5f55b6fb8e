// Host-loop stand-ins for the device primitives of the decoder backward, so
// that the schedule in bptt_plan.h (host logic: step order, the window's
// query-side records, step blocks, detach points, transposed operands,
// workspace layout) can be
// checked against the float64 oracle without a GPU.  Test infrastructure:
// the library never uses it.  Each member restates the specification of the
// kernel of the same name in bptt.cuh, in double arithmetic over fp32
// storage, with the storage-type writes optionally rounded to bf16 as the
// device's bf16 models round them.
#include "../recurrent_looped_transformer_rlt_b300/csrc/bptt_plan.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

namespace {

double sigm(double x) { return 1.0 / (1.0 + std::exp(-x)); }

// Round to the nearest bfloat16 (ties to even), kept as a float: the values
// a bf16 model stores in its storage-type buffers.
float bf16_round(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if ((u & 0x7f800000u) != 0x7f800000u) u = (u + 0x7fffu + ((u >> 16) & 1u)) & 0xffff0000u;
  memcpy(&x, &u, 4);
  return x;
}

void rope_cs(int p, int i, int hd, float theta, double& c, double& s) {
  const double a = p * std::pow((double)theta, -2.0 * i / hd);
  c = std::cos(a);
  s = std::sin(a);
}

struct HostOps {
  using T = float;
  bool bf16 = false;  // storage-type writes rounded to bf16 (the device's bf16 models)
  float st(double v) const { return bf16 ? bf16_round((float)v) : (float)v; }

  int zero(void* p, size_t bytes) {
    memset(p, 0, bytes);
    return 0;
  }
  int copy(void* dst, const void* src, size_t bytes) {
    memmove(dst, src, bytes);
    return 0;
  }
  int transpose(const T* src, int rows, int cols, int lds, T* dst, int ldd) {
    for (int r = 0; r < rows; ++r)
      for (int c = 0; c < cols; ++c) dst[(size_t)c * ldd + r] = src[(size_t)r * lds + c];
    return 0;
  }
  // C[M][N] (+)= A[M][K] W[N][K]^T
  int gemm(const T* A, int lda, int M, int K, const T* W, int ldw, int N, float* C, int ldc, bool add) {
    for (int m = 0; m < M; ++m)
      for (int n = 0; n < N; ++n) {
        double acc = 0;
        for (int k = 0; k < K; ++k) acc += (double)A[(size_t)m * lda + k] * W[(size_t)n * ldw + k];
        float& c = C[(size_t)m * ldc + n];
        c = add ? c + (float)acc : (float)acc;
      }
    return 0;
  }
  // C[M][N] = R[M][N] + A[M][K] W[N][K]^T (a residual update into a new buffer)
  int gemm_res(const T* A, int lda, int M, int K, const T* W, int ldw, int N, const float* R, float* C, int ldc) {
    for (int m = 0; m < M; ++m)
      for (int n = 0; n < N; ++n) {
        double acc = 0;
        for (int k = 0; k < K; ++k) acc += (double)A[(size_t)m * lda + k] * W[(size_t)n * ldw + k];
        C[(size_t)m * ldc + n] = R[(size_t)m * ldc + n] + (float)acc;
      }
    return 0;
  }
  // dm = A W^T, then the SwiGLU backward of every element into dY [B][2f]
  // (and transposed)
  int gemm_swiglu_bwd(const T* A, int lda, int M, int K, const T* W, int ldw, int f, const float* g, const float* u,
                      T* dY, T* dYT, int ldT) {
    std::vector<float> dm((size_t)M * f);
    gemm(A, lda, M, K, W, ldw, f, dm.data(), f, false);
    return swiglu_bwd(dm.data(), g, u, M, f, dY, dYT, ldT);
  }
  // d[e; s] = A W_g (columns < d to the e gradient row p, the rest to ds)
  int gemm_merge_bwd(const T* A, int lda, int M, int K, const T* W, int ldw, int d, int T_mem, const int* pos,
                     float* de, float* ds) {
    const int p = *pos;
    std::vector<float> dx((size_t)M * 2 * d);
    gemm(A, lda, M, K, W, ldw, 2 * d, dx.data(), 2 * d, false);
    return merge_bwd2(dx.data(), M, d, T_mem, p, de, ds);
  }
  int bcast_rows(float* dst, const float* src, int rows, int d) {
    for (int r = 0; r < rows; ++r) memcpy(dst + (size_t)r * d, src, sizeof(float) * d);
    return 0;
  }
  // position-dependent operands are read from the position cell *pos
  int merge_in(const T* e, int T_mem, const int* pos, const float* s_all, int B, int d, T* xg, T* xgT, int ldT) {
    const int p = *pos;
    const float* s = s_all + (size_t)p * B * d;
    for (int b = 0; b < B; ++b)
      for (int i = 0; i < 2 * d; ++i) {
        const float v = i < d ? e[((size_t)b * T_mem + p) * d + i] : st(s[(size_t)b * d + i - d]);
        xg[(size_t)b * 2 * d + i] = v;
        if (xgT) xgT[(size_t)i * ldT + b] = v;
      }
    return 0;
  }
  int merge_out(const float* zpre, const float* bg, const T* e, int T_mem, const int* pos, const float* s_all, int B,
                int d, float* z, float* h) {
    const int p = *pos;
    const float* s = s_all + (size_t)p * B * d;
    for (int b = 0; b < B; ++b)
      for (int i = 0; i < d; ++i) {
        const size_t o = (size_t)b * d + i;
        const double zv = zpre ? sigm((double)zpre[o] + bg[i]) : 0.0;
        const double ev = e[((size_t)b * T_mem + p) * d + i];
        z[o] = (float)zv;
        h[o] = (float)(zv * s[o] + (1 - zv) * ev);
      }
    return 0;
  }
  // x: rows [B][d], or with pos the rows of position (*pos + off) of [.][B][d]
  int rms_fwd(const float* x, const int* pos, int off, const float* g, int B, int d, float eps, float* r, T* y, T* yT,
              int ldT) {
    if (pos) x += (size_t)(*pos + off) * B * d;
    for (int b = 0; b < B; ++b) {
      const float* xr = x + (size_t)b * d;
      double ss = 0;
      for (int i = 0; i < d; ++i) ss += (double)xr[i] * xr[i];
      const double rv = 1.0 / std::sqrt(ss / d + eps);
      r[b] = (float)rv;
      for (int i = 0; i < d; ++i) {
        const float v = st(xr[i] * rv * g[i]);
        y[(size_t)b * d + i] = v;
        if (yT) yT[(size_t)i * ldT + b] = v;
      }
    }
    return 0;
  }
  void qkv_post(const float* qkv, int p, int B, int H, int hd, float theta, float* qo, T* K, T* V, int Tk) {
    const int d = H * hd, half = hd / 2;
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h)
        for (int i = 0; i < half; ++i) {
          double c, s;
          rope_cs(p, i, hd, theta, c, s);
          const float* row = qkv + (size_t)b * 3 * d + h * hd;
          float* q = qo + (size_t)b * d + h * hd;
          q[i] = (float)(row[i] * c - row[i + half] * s);
          q[i + half] = (float)(row[i + half] * c + row[i] * s);
          const size_t o = (((size_t)b * H + h) * Tk + p) * hd;
          K[o + i] = st(row[d + i] * c - row[d + i + half] * s);
          K[o + i + half] = st(row[d + i + half] * c + row[d + i] * s);
          V[o + i] = st(row[2 * d + i]);
          V[o + i + half] = st(row[2 * d + i + half]);
        }
  }
  // attention of q over positions j0..j1 (lse, output rows; oT optional)
  void attend(const float* q, const T* K, const T* V, int Tk, int j0, int j1, int B, int H, int hd, float scale,
              float* lse, T* oq, T* oT, int ldT) {
    const int d = H * hd;
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h) {
        const T* Kb = K + ((size_t)b * H + h) * Tk * hd;
        const T* Vb = V + ((size_t)b * H + h) * Tk * hd;
        const float* qq = q + (size_t)b * d + h * hd;
        std::vector<double> sc;
        for (int j = j0; j <= j1; ++j) {
          double a2 = 0;
          for (int i = 0; i < hd; ++i) a2 += (double)qq[i] * Kb[(size_t)j * hd + i];
          sc.push_back(a2 * scale);
        }
        const double mx = *std::max_element(sc.begin(), sc.end());
        double l = 0;
        for (double v : sc) l += std::exp(v - mx);
        const double ls = mx + std::log(l);
        lse[b * H + h] = (float)ls;
        for (int i = 0; i < hd; ++i) {
          double acc = 0;
          for (int j = j0; j <= j1; ++j) acc += std::exp(sc[j - j0] - ls) * Vb[(size_t)j * hd + i];
          const size_t c = (size_t)h * hd + i;
          oq[(size_t)b * d + c] = st(acc);
          if (oT) oT[c * ldT + b] = st(acc);
        }
      }
  }
  // memory attention of position p = *pos over positions 0..p: the LSE and
  // the output to the records (row p of [n][L] at lse_l, o_l with L rows per
  // position) and the output to o_step
  int attn_fwd(const float* q, const T* K, const T* V, int Tk, const int* pos, int /* n: the device's split grid */,
               int B, int H, int hd, float scale, float* lse_l, T* o_l, int L, T* o_step,
               float* /* scratch of the device's key split */) {
    const int p = *pos, d = H * hd;
    attend(q, K, V, Tk, 0, p, B, H, hd, scale, lse_l + (size_t)p * L * B * H, o_step, nullptr, 0);
    memcpy(o_l + (size_t)p * L * B * d, o_step, sizeof(T) * (size_t)B * d);
    return 0;
  }
  // window attention forward of position p = *pos: RoPE of q and k at p (q to
  // its record slot p mod W of qR, k and v to K/V at p), then the attention
  // over positions max(0, p - W + 1)..p (LSE to the record slot of lR)
  int swa_fwd(const float* qkv, const int* pos, int W, int B, int H, int hd, float theta, float scale, float* qR,
              float* lR, T* K, T* V, int Tk, T* oq, T* oT, int ldT, float* /* scratch of the device's key split */) {
    const int p = *pos, j0 = p - W + 1 > 0 ? p - W + 1 : 0;
    float* qo = qR + (size_t)(p % W) * B * H * hd;
    qkv_post(qkv, p, B, H, hd, theta, qo, K, V, Tk);
    attend(qo, K, V, Tk, j0, p, B, H, hd, scale, lR + (size_t)(p % W) * B * H, oq, oT, ldT);
    return 0;
  }
  // row p (L rows per position) of a recorded [n][L][B][N] operand into the
  // fixed rows y and the column slot yT
  int tcopy(const T* x_l, int L, const int* pos, int B, int N, T* y, T* yT, int ldT) {
    const T* x = x_l + (size_t)(*pos) * L * B * N;
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < N; ++j) {
        y[(size_t)b * N + j] = x[(size_t)b * N + j];
        yT[(size_t)j * ldT + b] = x[(size_t)b * N + j];
      }
    return 0;
  }
  int put_row(float* dst, const int* pos, int off, const float* src, int count) {
    memcpy(dst + (size_t)(*pos + off) * count, src, sizeof(float) * count);
    return 0;
  }
  int set_pos(int* pos, int v) {
    *pos = v;
    return 0;
  }
  int add_pos(int* pos, int dv) {
    *pos += dv;
    return 0;
  }
  template <class Fn>
  int step(int /* key of the device's captured step */, Fn fn) {
    return fn();
  }
  int zero_if_detached(float* ds, const int* pos, int s_every, int count) {
    const int p = *pos;
    if (p >= 1 && s_every > 0 && p % s_every == 0) memset(ds, 0, sizeof(float) * count);
    return 0;
  }
  int swiglu_fwd(const float* g, const float* u, int B, int f, T* m, T* mT, int ldT) {
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < f; ++j) {
        const size_t o = (size_t)b * f + j;
        const double gv = g[o];
        const float v = st(gv * sigm(gv) * u[o]);
        m[o] = v;
        if (mT) mT[(size_t)j * ldT + b] = v;
      }
    return 0;
  }
  int head_bwd(const float* logits, int B, int V, const int32_t* actions, int n, const int* pos, float inv_temp,
               int top_k, float* lp, T* dl, T* dlT, int ldT) {
    const int p = *pos;
    for (int b = 0; b < B; ++b) {
      std::vector<double> x(V);
      for (int v = 0; v < V; ++v) x[v] = (double)logits[(size_t)b * V + v] * inv_temp;
      std::vector<char> in(V, 1);
      if (top_k > 0 && top_k < V) {  // the k largest, ties to the lower id
        std::vector<int> id(V);
        std::iota(id.begin(), id.end(), 0);
        std::stable_sort(id.begin(), id.end(), [&](int a, int c) { return x[a] > x[c]; });
        std::fill(in.begin(), in.end(), 0);
        for (int r = 0; r < top_k; ++r) in[id[r]] = 1;
      }
      double mx = -1e300, se = 0;
      for (int v = 0; v < V; ++v)
        if (in[v]) mx = std::max(mx, x[v]);
      for (int v = 0; v < V; ++v)
        if (in[v]) se += std::exp(x[v] - mx);
      const double ls = mx + std::log(se);
      int a = actions[(size_t)b * n + p];
      if (a >= V) a = -1;
      const bool ain = a >= 0 && in[a];
      lp[(size_t)b * n + p] = a < 0 ? NAN : (ain ? (float)(x[a] - ls) : -INFINITY);
      for (int v = 0; v < V; ++v) {
        double gv = 0;
        if (a >= 0) gv = inv_temp * ((in[v] ? std::exp(x[v] - ls) : 0.0) - ((v == a && ain) ? 1.0 : 0.0));
        dl[(size_t)b * V + v] = st(gv);
        dlT[(size_t)v * ldT + b] = st(gv);
      }
    }
    return 0;
  }
  // dx += RMSNorm backward, dg += the gain gradient; with y given, the
  // updated dx rows also go to y (storage type) and yT (transposed)
  int rms_bwd(const float* x, const int* pos, int off, const float* r, const float* g, const float* dy, int B, int d,
              float* dx, float* dg, T* y, T* yT, int ldT) {
    if (pos) x += (size_t)(*pos + off) * B * d;
    for (int i = 0; i < d; ++i) {
      double acc = 0;
      for (int b = 0; b < B; ++b) acc += (double)dy[(size_t)b * d + i] * x[(size_t)b * d + i] * r[b];
      dg[i] += (float)acc;
    }
    for (int b = 0; b < B; ++b) {
      const float* xr = x + (size_t)b * d;
      const float* dyr = dy + (size_t)b * d;
      double sd = 0;
      for (int i = 0; i < d; ++i) sd += (double)g[i] * dyr[i] * xr[i];
      const double rv = r[b], coef = rv * rv * rv * sd / d;
      for (int i = 0; i < d; ++i) {
        float& v = dx[(size_t)b * d + i];
        v += (float)(rv * g[i] * dyr[i] - xr[i] * coef);
        if (y) {
          y[(size_t)b * d + i] = st(v);
          yT[(size_t)i * ldT + b] = st(v);
        }
      }
    }
    return 0;
  }
  int pack(const float* x, int B, int N, T* y, T* yT, int ldT) {
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < N; ++j) {
        y[(size_t)b * N + j] = st(x[(size_t)b * N + j]);
        yT[(size_t)j * ldT + b] = st(x[(size_t)b * N + j]);
      }
    return 0;
  }
  int swiglu_bwd(const float* dm, const float* g, const float* u, int B, int f, T* dY, T* dYT, int ldT) {
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < f; ++j) {
        const size_t o = (size_t)b * f + j;
        const double gv = g[o], uv = u[o], dv = dm[o], sg = sigm(gv);
        const float dgv = st(dv * uv * sg * (1 + gv * (1 - sg))), duv = st(dv * gv * sg);
        dY[(size_t)b * 2 * f + j] = dgv;
        dY[(size_t)b * 2 * f + f + j] = duv;
        dYT[(size_t)j * ldT + b] = dgv;
        dYT[(size_t)(f + j) * ldT + b] = duv;
      }
    return 0;
  }
  // dq of the attention over positions j0..j1 (fp32 [B][d]), D = g.o from the
  // stored output o (written to Dout when given)
  void attn_dq(const float* q, const float* gout, const T* o, const float* lse, const T* K, const T* V, int Tk, int j0,
               int j1, int B, int H, int hd, float scale, float* dq, float* Dout) {
    const int d = H * hd;
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h) {
        const float* qq = q + (size_t)b * d + h * hd;
        const float* gg = gout + (size_t)b * d + h * hd;
        const T* oo = o + (size_t)b * d + h * hd;
        const T* Kb = K + ((size_t)b * H + h) * Tk * hd;
        const T* Vb = V + ((size_t)b * H + h) * Tk * hd;
        double D = 0;
        for (int i = 0; i < hd; ++i) D += (double)gg[i] * oo[i];
        if (Dout) Dout[b * H + h] = (float)D;
        std::vector<double> acc(hd, 0.0);
        for (int j = j0; j <= j1; ++j) {
          double s = 0, dp = 0;
          for (int i = 0; i < hd; ++i) {
            s += (double)qq[i] * Kb[(size_t)j * hd + i];
            dp += (double)gg[i] * Vb[(size_t)j * hd + i];
          }
          const double P = std::exp(s * scale - lse[b * H + h]), dS = P * (dp - D);
          for (int i = 0; i < hd; ++i) acc[i] += dS * Kb[(size_t)j * hd + i];
        }
        for (int i = 0; i < hd; ++i) dq[(size_t)b * d + h * hd + i] = (float)(scale * acc[i]);
      }
  }
  // the query gradient of the memory attention of position p = *pos (LSE
  // row p of lse_l with L rows per position), written as the next
  // projection's operands (storage type [B][d] and transposed)
  int attn_bwd(const float* q, const float* gout, const T* o, const float* lse_l, int L, const T* K, const T* V, int Tk,
               const int* pos, int /* n: the device's split grid */, int B, int H, int hd, float scale, float* Dout,
               T* dqY, T* dqT, int ldT, float* /* scratch of the device's key split */) {
    const int p = *pos, d = H * hd;
    std::vector<float> dq((size_t)B * d);
    attn_dq(q, gout, o, lse_l + (size_t)p * L * B * H, K, V, Tk, 0, p, B, H, hd, scale, dq.data(), Dout);
    return pack(dq.data(), B, d, dqY, dqT, ldT);
  }
  // key/value gradient of window position p from the query-side records of
  // positions p..p_last (ring slot p' mod W of one layer: q, g [W][B][d],
  // lse, D [W][B][H]) into dK, dV [B][d]
  void kv_grad(const T* K, const T* V, int Tk, int p, int p_last, const float* qR, const float* gR, const float* lR,
               const float* DR, int W, int B, int H, int hd, float scale, float* dK, float* dV) {
    const int d = H * hd;
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h) {
        const T* kp = K + (((size_t)b * H + h) * Tk + p) * hd;
        const T* vp = V + (((size_t)b * H + h) * Tk + p) * hd;
        std::vector<double> ak(hd, 0.0), av(hd, 0.0);
        for (int pp = p; pp <= p_last; ++pp) {
          const size_t row = (size_t)(pp % W) * B + b;
          const float* qq = qR + row * d + h * hd;
          const float* gg = gR + row * d + h * hd;
          double sc = 0, dp = 0;
          for (int i = 0; i < hd; ++i) {
            sc += (double)qq[i] * kp[i];
            dp += (double)gg[i] * vp[i];
          }
          const double P = std::exp(sc * scale - lR[row * H + h]), dS = P * (dp - DR[row * H + h]);
          for (int i = 0; i < hd; ++i) {
            ak[i] += scale * dS * qq[i];
            av[i] += P * gg[i];
          }
        }
        for (int i = 0; i < hd; ++i) {
          dK[(size_t)b * d + h * hd + i] = (float)ak[i];
          dV[(size_t)b * d + h * hd + i] = (float)av[i];
        }
      }
  }
  // memory gradient of one block: for every position j <= p_hi, the steps
  // s < nb of the block (position p_hi - s >= j) and the layers [l0, l1)
  int mem_grad(const T* K, const T* V, int T_mem, const float* qS, const float* gS, const float* lse_all,
               const float* DS, int L, int l0, int l1, int nb, int p_hi, int B, int H, int hd, float scale, float* dK,
               float* dV) {
    const int d = H * hd;
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h)
        for (int j = 0; j <= p_hi; ++j) {
          const T* kj = K + (((size_t)b * H + h) * T_mem + j) * hd;
          const T* vj = V + (((size_t)b * H + h) * T_mem + j) * hd;
          std::vector<double> ak(hd, 0.0), av(hd, 0.0);
          for (int s = 0; s < nb && p_hi - s >= j; ++s)
            for (int l = l0; l < l1; ++l) {
              const size_t row = ((size_t)s * L + l) * B + b;
              const float* qq = qS + row * d + h * hd;
              const float* gg = gS + row * d + h * hd;
              const double ls = lse_all[(((size_t)(p_hi - s) * L + l) * B + b) * H + h];
              const double Dv = DS[row * H + h];
              double sc = 0, dp = 0;
              for (int i = 0; i < hd; ++i) {
                sc += (double)qq[i] * kj[i];
                dp += (double)gg[i] * vj[i];
              }
              const double P = std::exp(sc * scale - ls), dS = P * (dp - Dv);
              for (int i = 0; i < hd; ++i) {
                ak[i] += scale * dS * qq[i];
                av[i] += P * gg[i];
              }
            }
          const size_t base = (((size_t)b * H + h) * T_mem + j) * hd;
          for (int i = 0; i < hd; ++i) {
            dK[base + i] += (float)ak[i];
            dV[base + i] += (float)av[i];
          }
        }
    return 0;
  }
  // d qkv of position p: dq and dK back through RoPE, dV as is
  void qkv_bwd(const float* dq, const float* dK, const float* dV, int p, int B, int H, int hd, float theta, T* dY,
               T* dYT, int ldT) {
    const int d = H * hd, half = hd / 2;
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h)
        for (int i = 0; i < half; ++i) {
          double c, s;
          rope_cs(p, i, hd, theta, c, s);
          const size_t o = (size_t)b * d + h * hd;
          const double q1 = dq[o + i], q2 = dq[o + i + half];
          const double k1 = dK[o + i], k2 = dK[o + i + half], v1 = dV[o + i], v2 = dV[o + i + half];
          const double vals[6] = {q1 * c + q2 * s, -q1 * s + q2 * c, k1 * c + k2 * s, -k1 * s + k2 * c, v1, v2};
          const int cols[6] = {h * hd + i,     h * hd + i + half,     d + h * hd + i,
                               d + h * hd + i + half, 2 * d + h * hd + i, 2 * d + h * hd + i + half};
          for (int j = 0; j < 6; ++j) {
            dY[(size_t)b * 3 * d + cols[j]] = st(vals[j]);
            dYT[(size_t)cols[j] * ldT + b] = st(vals[j]);
          }
        }
  }
  // window attention backward of position p = *pos (one layer): this step's
  // output gradient g into its record (slot p mod W), the query gradient over
  // positions max(0, p - W + 1)..p (D written to the record), the key/value
  // gradient of position p from the records of positions p..p_last (p_last =
  // p with the cache detached, else min(p + W - 1, n - 1); n = Tk), both back
  // through RoPE, the value gradient as is, into d qkv [B][3d] (storage type,
  // and transposed)
  int swa_bwd(const T* K, const T* V, int Tk, const int* pos, int W, bool cache, const T* o, const float* g,
              float* qR, float* gR, float* lR, float* DR, int B, int H, int hd, float scale, float theta, T* dY, T* dYT,
              int ldT, float* /* scratch of the device's split */) {
    const int p = *pos, j0 = p - W + 1 > 0 ? p - W + 1 : 0;
    const int p_last = cache ? p : (p + W - 1 < Tk - 1 ? p + W - 1 : Tk - 1);
    const size_t Bd = (size_t)B * H * hd, BH = (size_t)B * H, r = (size_t)(p % W);
    memcpy(gR + r * Bd, g, sizeof(float) * Bd);
    std::vector<float> dq(Bd), dK(Bd), dV(Bd);
    attn_dq(qR + r * Bd, gR + r * Bd, o, lR + r * BH, K, V, Tk, j0, p, B, H, hd, scale, dq.data(), DR + r * BH);
    kv_grad(K, V, Tk, p, p_last, qR, gR, lR, DR, W, B, H, hd, scale, dK.data(), dV.data());
    qkv_bwd(dq.data(), dK.data(), dV.data(), p, B, H, hd, theta, dY, dYT, ldT);
    return 0;
  }
  int merge_bwd(const float* dh, const float* z, const T* e, int T_mem, const int* pos, const float* s_all, int B,
                int d, bool gate, T* dY, T* dYT, int ldT, float* dbg, float* de, float* ds) {
    const int p = *pos;
    const float* s = s_all + (size_t)p * B * d;
    for (int i = 0; i < d; ++i) {
      double acc = 0;
      for (int b = 0; b < B; ++b) {
        const size_t o = (size_t)b * d + i, oe = ((size_t)b * T_mem + p) * d + i;
        const double g = dh[o], zv = z[o];
        if (de) de[oe] = (float)(g * (1 - zv));
        ds[o] = (float)(g * zv);
        if (gate) {
          const double dz = g * (s[o] - e[oe]) * zv * (1 - zv);
          dY[o] = st(dz);
          dYT[(size_t)i * ldT + b] = st(dz);
          acc += dz;
        }
      }
      if (gate) dbg[i] += (float)acc;
    }
    return 0;
  }
  int merge_bwd2(const float* dx, int B, int d, int T_mem, int p, float* de, float* ds) {
    for (int b = 0; b < B; ++b)
      for (int i = 0; i < d; ++i) {
        if (de) de[((size_t)b * T_mem + p) * d + i] += dx[(size_t)b * 2 * d + i];
        ds[(size_t)b * d + i] += dx[(size_t)b * 2 * d + d + i];
      }
    return 0;
  }
  int colsum(const float* x, int B, int d, float* out) {
    for (int i = 0; i < d; ++i) {
      double a = 0;
      for (int b = 0; b < B; ++b) a += x[(size_t)b * d + i];
      out[i] += (float)a;
    }
    return 0;
  }
  int loss_sum(const float* lp, const int32_t* actions, int B, int n, int V, float* loss) {
    double a = 0;
    for (size_t i = 0; i < (size_t)B * n; ++i)
      if (actions[i] >= 0 && actions[i] < V) a -= lp[i];
    *loss = (float)a;
    return 0;
  }
};

}  // namespace

// sh: B n T_mem d H hd f L W V G gate_learned top_k detach_s_every detach_cache detach_memory S bf16
// fp: rms_eps rope_theta temperature
// P (in order): W_g W_qkv W_O W_Qx W_Ox W_1 W_3 W_2 W_o b_g s_star dec_attn_norm dec_xattn_norm dec_ffn_norm
//   head_norm | e mem actions | loss logp | gradients in rlt_grads order | d_e d_mem
extern "C" int bptt_host(const int* sh, const float* fp, void** P) {
  bpplan::Shape S{};
  S.B = sh[0];
  S.n = sh[1];
  S.T_mem = sh[2];
  S.d = sh[3];
  S.H = sh[4];
  S.hd = sh[5];
  S.f = sh[6];
  S.L = sh[7];
  S.W = sh[8];
  S.V = sh[9];
  S.G = sh[10];
  S.gate_learned = sh[11] != 0;
  S.top_k = sh[12];
  S.eps = fp[0];
  S.theta = fp[1];
  S.scale = 1.0f / std::sqrt((float)S.hd);
  S.inv_temp = 1.0f / fp[2];
  S.Bp = S.B;
  S.S = sh[16];
  S.chunk = 0;
  const bool bf16 = sh[17] != 0;
  const bpplan::Detach D{sh[13], sh[14] != 0, sh[15] != 0};
  auto cf = [&](int i) { return static_cast<const float*>(P[i]); };
  auto mf = [&](int i) { return static_cast<float*>(P[i]); };
  const bpplan::Params<float> Pp{cf(0), cf(1), cf(2),  cf(3),  cf(4),  cf(5),  cf(6), cf(7),
                                 cf(8), cf(9), cf(10), cf(11), cf(12), cf(13), cf(14)};
  const bpplan::Io<float> io{cf(15), cf(16), static_cast<const int32_t*>(P[17]), mf(18), mf(19), mf(35), mf(36)};
  const bpplan::Grads G{mf(20), mf(21), mf(22), mf(23), mf(24), mf(25), mf(26), mf(27),
                        mf(28), mf(29), mf(30), mf(31), mf(32), mf(33), mf(34)};
  const bpplan::Layout Lw = bpplan::layout(S, sizeof(float), 256);
  std::vector<double> ws((Lw.total + 7) / 8);  // 8-byte aligned storage
  HostOps k;
  k.bf16 = bf16;
  return bpplan::run(k, S, D, Pp, io, G, reinterpret_cast<char*>(ws.data()), Lw);
}
