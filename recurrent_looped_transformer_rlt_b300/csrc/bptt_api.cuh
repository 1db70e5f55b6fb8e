// Backpropagation through time of the decoder (rlt_bptt_workspace_size,
// rlt_bptt in include/rlt.h): the operations of bptt_plan.h as launches on
// one CUDA stream.  Part of the rlt_api.cu translation unit (included at its
// end): the projections go through the same launchers as the forward step -
// tcgen05 weight streaming for bf16 models, the fp32 CUDA-core kernel for
// fp32 models.
#include "bptt.cuh"
#include "bptt_plan.h"

namespace {

template <typename T_>
struct BpttOps {
  using T = T_;
  static constexpr bool kBf16 = std::is_same<T_, bf16>::value;
  cudaStream_t st;   // the stream launches go to (the capture stream while capturing)
  cudaStream_t user; // the caller's stream (graphs are replayed on it)
  cudaStream_t cap;  // the model's capture stream
  bool graphs = true;
  bool mg_tc = true;  // bf16 models: the memory gradient on the tensor cores (mem_grad_tc_kernel)
  TcScratch sc;
  int* status;
  // one captured step per key: -1 the recording step, s >= 0 the reverse
  // step of block slot s
  struct Step {
    int key;
    cudaGraphExec_t exec;
    uint64_t launches;
  };
  std::vector<Step> steps;

  ~BpttOps() {
    for (auto& x : steps) cudaGraphExecDestroy(x.exec);
  }
  int post() {
    g_launches++;
    return launch_ok();
  }
  static unsigned blocks(size_t work, int per_block = bptt::kThreads) { return cdiv(work, per_block); }
  static int splits(int range) { return (range + bptt::kAttnChunk - 1) / bptt::kAttnChunk; }

  // Runs fn's launches as one step: captured on the first call of a key into
  // a graph, replayed on the caller's stream from then on (the launches read
  // the step's position from the device cell, so every replay is the step at
  // the cell's current position).
  template <class Fn>
  int step(int key, Fn fn) {
    if (!graphs) return fn();
    for (auto& x : steps)
      if (x.key == key) {
        if (cudaGraphLaunch(x.exec, user) != cudaSuccess) return RLT_ECUDA;
        g_launches += x.launches;
        return RLT_OK;
      }
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    // the capture stream starts after the caller's stream's earlier work
    RLT_CUDA_TRY(cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal));
    const uint64_t before = g_launches.load();
    st = cap;
    int rc = fn();
    st = user;
    const uint64_t nk = g_launches.load() - before;
    g_launches.store(before);
    const cudaError_t ce = cudaStreamEndCapture(cap, &graph);
    if (rc) {
      if (graph) cudaGraphDestroy(graph);
      return rc;
    }
    if (ce != cudaSuccess) return RLT_ECUDA;
    const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) return RLT_ECUDA;
    steps.push_back({key, exec, nk});
    if (cudaGraphLaunch(exec, user) != cudaSuccess) return RLT_ECUDA;
    g_launches += nk;
    return RLT_OK;
  }

  int zero(void* p, size_t bytes) {
    if (!bytes) return RLT_OK;
    return cudaMemsetAsync(p, 0, bytes, st) == cudaSuccess ? RLT_OK : RLT_ECUDA;
  }
  int copy(void* dst, const void* src, size_t bytes) {
    if (!bytes) return RLT_OK;
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st) == cudaSuccess ? RLT_OK : RLT_ECUDA;
  }
  int set_pos(int* pos, int v) {
    bptt::set_pos_kernel<<<1, 1, 0, st>>>(pos, v);
    return post();
  }
  int add_pos(int* pos, int dv) {
    bptt::add_pos_kernel<<<1, 1, 0, st>>>(pos, dv);
    return post();
  }
  int put_row(float* dst, const int* pos, int off, const float* src, int count) {
    bptt::put_row_kernel<<<blocks((size_t)count), bptt::kThreads, 0, st>>>(dst, pos, off, src, count);
    return post();
  }
  int zero_if_detached(float* ds, const int* pos, int s_every, int count) {
    bptt::zero_if_detached_kernel<<<blocks((size_t)count), bptt::kThreads, 0, st>>>(ds, pos, s_every, count);
    return post();
  }
  int transpose(const T* src, int rows, int cols, int lds, T* dst, int ldd) {
    bptt::transpose_kernel<T><<<dim3(cdiv(cols, 32), cdiv(rows, 32)), dim3(32, 8), 0, st>>>(src, rows, cols, lds,
                                                                                           dst, ldd);
    return post();
  }
  // C[M][N] (+)= A[M][K] W[N][K]^T
  int gemm(const T* A, int lda, int M, int K, const T* W_, int ldw, int N, float* C, int ldc, bool add) {
    if (add) return gemm_epi(A, lda, M, K, W_, ldw, N, EpiAddF32{C, ldc});
    return gemm_epi(A, lda, M, K, W_, ldw, N, EpiStoreF32{C, ldc});
  }
  // A[M][K] W[N][K]^T through the epilogue functor
  template <class Epi>
  int gemm_epi(const T* A, int lda, int M, int K, const T* W_, int ldw, int N, Epi epi) {
    if constexpr (kBf16) {
      AArg a;
      a.A = A;
      a.lda = lda;
      return proj_bf16<false>(st, a, M, K, W_, nullptr, ldw, N, epi, sc);
    } else {
      return ::gemm<float>(st, A, lda, GemmB{W_, W_, N, ldw}, M, N, K, epi);
    }
  }
  // C[M][N] = R[M][N] + A[M][K] W[N][K]^T
  int gemm_res(const T* A, int lda, int M, int K, const T* W_, int ldw, int N, const float* R, float* C, int ldc) {
    return gemm_epi(A, lda, M, K, W_, ldw, N, bptt::EpiResidualInto{R, C, ldc});
  }
  // dm = A W^T, SwiGLU backward in the epilogue into dY [M][2f] and dYT
  int gemm_swiglu_bwd(const T* A, int lda, int M, int K, const T* W_, int ldw, int f, const float* g, const float* u,
                      T* dY, T* dYT, int ldT) {
    return gemm_epi(A, lda, M, K, W_, ldw, f, bptt::EpiSwigluBwd<T>{g, u, f, dY, dYT, ldT});
  }
  // d[e; s] = dzpre W_g (A = dzpre, W = the transposed copy of W_g), added to
  // the e gradient of position *pos and to ds
  int gemm_merge_bwd(const T* A, int lda, int M, int K, const T* W_, int ldw, int d, int T_mem, const int* pos,
                     float* de, float* ds) {
    return gemm_epi(A, lda, M, K, W_, ldw, 2 * d, bptt::EpiMergeBwd{de, ds, d, T_mem, pos});
  }
  int bcast_rows(float* dst, const float* src, int rows, int d) {
    bcast_rows_kernel<<<blocks((size_t)rows * d), bptt::kThreads, 0, st>>>(dst, src, rows, d);
    return post();
  }
  int merge_in(const T* e, int T_mem, const int* pos, const float* s_all, int B, int d, T* xg, T* xgT, int ldT) {
    bptt::merge_in_kernel<T><<<blocks((size_t)B * 2 * d), bptt::kThreads, 0, st>>>(e, T_mem, pos, s_all, B, d, xg,
                                                                                  xgT, ldT);
    return post();
  }
  int merge_out(const float* zpre, const float* bg, const T* e, int T_mem, const int* pos, const float* s_all, int B,
                int d, float* z, float* h) {
    bptt::merge_out_kernel<T><<<blocks((size_t)B * d), bptt::kThreads, 0, st>>>(zpre, bg, e, T_mem, pos, s_all, B, d,
                                                                              z, h);
    return post();
  }
  int rms_fwd(const float* x, const int* pos, int off, const float* g, int B, int d, float eps, float* r, T* y, T* yT,
              int ldT) {
    bptt::rms_fwd_kernel<T><<<blocks((size_t)B * 32), bptt::kThreads, 0, st>>>(x, pos, off, g, B, d, eps, r, y, yT,
                                                                              ldT);
    return post();
  }
  // window attention forward: one warp per (b, h) for windows of one chunk,
  // else split over the keys (grid sized for the full window) and combined
  int swa_fwd(const float* qkv, const int* pos, int Wn, int B, int H, int hd, float theta, float scale, float* qR,
              float* lR, T* K, T* V, int Tk, T* oq, T* oT, int ldT, float* part) {
    const int nsplit = splits(Wn);
    const size_t pairs = (size_t)B * H;
    if (nsplit <= 1) {
      bptt::swa_fwd_kernel<T><<<blocks(pairs * 32, 128), 128, 0, st>>>(qkv, pos, Wn, B, H, hd, theta, scale, qR, lR,
                                                                       K, V, Tk, oq, oT, ldT);
      return post();
    }
    bptt::swa_part_fwd_kernel<T><<<blocks(pairs * nsplit * 32, 128), 128, 0, st>>>(qkv, pos, Wn, B, H, hd, theta,
                                                                                   scale, nsplit, qR, K, V, Tk, part);
    int rc = post();
    if (rc) return rc;
    bptt::attn_combine_fwd_kernel<T><<<blocks(pairs * 32, 128), 128, 0, st>>>(
        part, nsplit, B, H, hd, pos, lR, pairs, Wn, oq, oT, ldT, static_cast<T*>(nullptr), 0);
    return post();
  }
  // memory attention of the position in the cell over positions 0..p: one
  // warp per (b, h) when the call's steps fit one chunk, else split over the
  // keys (grid sized for the call's last position) and combined
  int attn_fwd(const float* q, const T* K, const T* V, int Tk, const int* pos, int n, int B, int H, int hd,
               float scale, float* lse_l, T* o_l, int L, T* o_step, float* part) {
    const int nsplit = splits(n);
    const size_t pairs = (size_t)B * H, d = (size_t)H * hd;
    if (nsplit <= 1) {
      bptt::attn_fwd_kernel<T><<<blocks(pairs * 32, 128), 128, 0, st>>>(q, K, V, Tk, pos, B, H, hd, scale, lse_l,
                                                                        (size_t)L * pairs, o_step, o_l,
                                                                        (size_t)L * B * d);
      return post();
    }
    bptt::attn_part_fwd_kernel<T><<<blocks(pairs * nsplit * 32, 128), 128, 0, st>>>(q, K, V, Tk, pos, B, H, hd,
                                                                                    scale, nsplit, part);
    int rc = post();
    if (rc) return rc;
    bptt::attn_combine_fwd_kernel<T><<<blocks(pairs * 32, 128), 128, 0, st>>>(
        part, nsplit, B, H, hd, pos, lse_l, (size_t)L * pairs, 0, o_step, static_cast<T*>(nullptr), 0, o_l,
        (size_t)L * B * d);
    return post();
  }
  int tcopy(const T* x_l, int L, const int* pos, int B, int N, T* y, T* yT, int ldT) {
    bptt::tcopy_kernel<T><<<blocks((size_t)B * N), bptt::kThreads, 0, st>>>(x_l, L, pos, B, N, y, yT, ldT);
    return post();
  }
  int swiglu_fwd(const float* g, const float* u, int B, int f, T* m, T* mT, int ldT) {
    bptt::swiglu_fwd_kernel<T><<<blocks((size_t)B * f), bptt::kThreads, 0, st>>>(g, u, B, f, m, mT, ldT);
    return post();
  }
  int head_bwd(const float* logits, int B, int V, const int32_t* actions, int n, const int* pos, float inv_temp,
               int top_k, float* lp, T* dl, T* dlT, int ldT) {
    bptt::head_bwd_kernel<<<B, bptt::kThreadsHead, sizeof(float) * (size_t)V, st>>>(
        logits, B, V, actions, n, pos, inv_temp, top_k, lp, dl, dlT, ldT, kBf16 ? 1 : 0, status);
    return post();
  }
  int rms_bwd(const float* x, const int* pos, int off, const float* r, const float* g, const float* dy, int B, int d,
              float* dx, float* dg, T* out, T* outT, int ldT) {
    const int row_blocks = (int)blocks((size_t)B * 32);
    const int col_blocks = (int)blocks((size_t)d);
    bptt::rms_bwd_kernel<T><<<row_blocks + col_blocks, bptt::kThreads, 0, st>>>(x, pos, off, r, g, dy, B, d, dx, dg,
                                                                               row_blocks, out, outT, ldT);
    return post();
  }
  int attn_bwd(const float* q, const float* gout, const T* o, const float* lse_l, int L, const T* K, const T* V,
               int Tk, const int* pos, int n, int B, int H, int hd, float scale, float* Dout, T* dqY, T* dqT, int ldT,
               float* part) {
    const int nsplit = splits(n);
    const size_t pairs = (size_t)B * H;
    if (nsplit <= 1) {
      bptt::attn_bwd_kernel<T><<<blocks(pairs * 32, 128), 128, 0, st>>>(q, gout, o, lse_l, (size_t)L * pairs, K, V,
                                                                        Tk, pos, B, H, hd, scale, Dout, dqY, dqT,
                                                                        ldT);
      return post();
    }
    bptt::attn_part_bwd_kernel<T><<<blocks(pairs * nsplit * 32, 128), 128, 0, st>>>(
        q, gout, o, lse_l, (size_t)L * pairs, K, V, Tk, pos, B, H, hd, scale, nsplit, part);
    int rc = post();
    if (rc) return rc;
    bptt::attn_combine_bwd_kernel<T><<<blocks(pairs * 32, 128), 128, 0, st>>>(part, nsplit, B, H, hd, scale, Dout,
                                                                             dqY, dqT, ldT);
    return post();
  }
  // window attention backward: one warp per (b, h) when the window fits one
  // chunk, else split over key and record chunks (grid sized for the full
  // window) and combined
  int swa_bwd(const T* K, const T* V, int Tk, const int* pos, int Wn, bool cache, const T* o, const float* g,
              float* qR, float* gR, float* lR, float* DR, int B, int H, int hd, float scale, float theta, T* dY,
              T* dYT, int ldT, float* part) {
    const int nsplit = splits(Wn);
    const size_t pairs = (size_t)B * H;
    if (nsplit <= 1) {
      bptt::swa_bwd_kernel<T><<<blocks(pairs * 32, 128), 128, 0, st>>>(
          K, V, Tk, pos, Wn, cache ? 1 : 0, o, g, qR, gR, lR, DR, B, H, hd, scale, theta, dY, dYT, ldT);
      return post();
    }
    bptt::swa_part_bwd_kernel<T><<<blocks(pairs * nsplit * 32, 128), 128, 0, st>>>(
        K, V, Tk, pos, Wn, cache ? 1 : 0, o, g, qR, gR, lR, DR, B, H, hd, scale, nsplit, part);
    int rc = post();
    if (rc) return rc;
    bptt::swa_combine_bwd_kernel<T><<<blocks(pairs * 32, 128), 128, 0, st>>>(part, nsplit, pos, Wn, B, H, hd, scale,
                                                                            theta, DR, dY, dYT, ldT);
    return post();
  }
  int mem_grad(const T* K, const T* V, int T_mem, const float* qS, const float* gS, const float* lse_all,
               const float* DS, int L, int l0, int l1, int nb, int p_hi, int B, int H, int hd, float scale, float* dK,
               float* dV) {
    if constexpr (kBf16) {
      if (mg_tc && (hd == 32 || hd == 64 || hd == 128)) {
        const dim3 g2(cdiv((size_t)p_hi + 1, bptt::kMgKeys), (unsigned)(B * H));
        if (hd == 32)
          bptt::mem_grad_tc_kernel<32><<<g2, bptt::kMgWarps * 32, 0, st>>>(K, V, T_mem, qS, gS, lse_all, DS, L, l0, l1,
                                                                           nb, p_hi, B, H, scale, dK, dV);
        else if (hd == 64)
          bptt::mem_grad_tc_kernel<64><<<g2, bptt::kMgWarps * 32, 0, st>>>(K, V, T_mem, qS, gS, lse_all, DS, L, l0, l1,
                                                                           nb, p_hi, B, H, scale, dK, dV);
        else
          bptt::mem_grad_tc_kernel<128><<<g2, bptt::kMgWarps * 32, 0, st>>>(K, V, T_mem, qS, gS, lse_all, DS, L, l0,
                                                                            l1, nb, p_hi, B, H, scale, dK, dV);
        return post();
      }
    }
    const dim3 grid(cdiv((size_t)p_hi + 1, bptt::kMemKeys), (unsigned)(B * H));
    bptt::mem_grad_kernel<T><<<grid, bptt::kMemWarps * 32, 0, st>>>(K, V, T_mem, qS, gS, lse_all, DS, L, l0, l1, nb,
                                                                    p_hi, B, H, hd, scale, dK, dV);
    return post();
  }
  int merge_bwd(const float* dh, const float* z, const T* e, int T_mem, const int* pos, const float* s_all, int B,
                int d, bool gate, T* dY, T* dYT, int ldT, float* dbg, float* de, float* ds) {
    bptt::merge_bwd_kernel<T><<<blocks((size_t)d), bptt::kThreads, 0, st>>>(dh, z, e, T_mem, pos, s_all, B, d,
                                                                            gate ? 1 : 0, dY, dYT, ldT, dbg, de, ds);
    return post();
  }
  int colsum(const float* x, int B, int d, float* out) {
    bptt::colsum_kernel<<<blocks((size_t)d), bptt::kThreads, 0, st>>>(x, B, d, out);
    return post();
  }
  int loss_sum(const float* lp, const int32_t* actions, int B, int n, int V, float* loss) {
    bptt::loss_sum_kernel<<<1, bptt::kThreads, 0, st>>>(lp, actions, B, n, V, loss);
    return post();
  }
};

constexpr size_t kBpttHeader = kWsHeaderBytes;
// steps per block: weight gradients are added by one GEMM over the block's
// S * B rows, and the memory gradient by one key-parallel pass per block
constexpr int kBpttBlock = 16;

bpplan::Shape bptt_shape(const rlt_model* m, int B, int n, int T_mem, float temperature, int top_k) {
  const rlt_config& c = m->cfg;
  bpplan::Shape S{};
  S.B = B;
  S.n = n;
  S.T_mem = T_mem;
  S.d = c.d_model;
  S.H = c.n_heads;
  S.hd = c.head_dim;
  S.f = c.d_ffn;
  S.L = c.n_layers;
  S.W = c.window;
  S.V = c.vocab;
  S.G = c.mem_groups;
  S.gate_learned = c.gate_mode == RLT_GATE_LEARNED;
  S.eps = c.rms_eps;
  S.theta = c.rope_theta;
  S.scale = 1.0f / sqrtf((float)c.head_dim);
  S.inv_temp = 1.0f / temperature;
  S.top_k = top_k;
  // the bf16 weight-gradient GEMMs contract over step slots of Bp rows in
  // whole 64-wide k-blocks
  S.Bp = (c.dtype == RLT_BF16) ? (B + 63) / 64 * 64 : B;
  S.S = n < kBpttBlock ? n : kBpttBlock;
  S.chunk = bptt::kAttnChunk;
  return S;
}

template <typename T_>
int bptt_impl(const rlt_model* m, const bpplan::Shape& S, const bpplan::Detach& D,
              const bpplan::Io<T_>& io, const bpplan::Grads& G, void* ws, cudaStream_t st, bool graphs,
              bool mg_tc) {
  const rlt_weights& w = m->w;
  bpplan::Params<T_> P;
  P.W_g = static_cast<const T_*>(w.W_g);
  P.W_qkv = static_cast<const T_*>(w.W_qkv);
  P.W_O = static_cast<const T_*>(w.W_O);
  P.W_Qx = static_cast<const T_*>(w.W_Qx);
  P.W_Ox = static_cast<const T_*>(w.W_Ox);
  P.W_1 = static_cast<const T_*>(w.W_1);
  P.W_3 = static_cast<const T_*>(w.W_3);
  P.W_2 = static_cast<const T_*>(w.W_2);
  P.W_o = static_cast<const T_*>(w.W_o);
  P.b_g = w.b_g;
  P.s_star = w.s_star;
  P.attn_norm = w.dec_attn_norm;
  P.xattn_norm = w.dec_xattn_norm;
  P.ffn_norm = w.dec_ffn_norm;
  P.head_norm = w.head_norm;
  const bpplan::Layout Lw = bpplan::layout(S, m->esz, kBpttHeader);
  BpttOps<T_> k;
  k.st = st;
  k.user = st;
  k.cap = m->cap_stream;
  k.graphs = graphs;
  k.mg_tc = mg_tc;
  k.status = static_cast<int*>(ws);
  k.sc.n_sm = m->n_sm;
  k.sc.maxc = m->gemm_maxc;
  k.sc.status = k.status;
  return bpplan::run(k, S, D, P, io, G, static_cast<char*>(ws), Lw);
}

bool g_bptt_attr_done = false;
std::mutex g_bptt_attr_mu;

int bptt_attrs() {
  std::lock_guard<std::mutex> lk(g_bptt_attr_mu);
  if (g_bptt_attr_done) return RLT_OK;
  // the head reduction keeps a row of V fp32 logits in shared memory
  const int smem = (int)sizeof(float) * 49152;
  if (cudaFuncSetAttribute(bptt::head_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return RLT_ECUDA;
  g_bptt_attr_done = true;
  return RLT_OK;
}

}  // namespace

extern "C" {

int rlt_bptt_workspace_size(const rlt_model* m, int32_t B, int32_t n, size_t* bytes) {
  if (!m || !bytes || B <= 0 || n <= 0) return RLT_EINVAL;
  *bytes = bpplan::layout(bptt_shape(m, B, n, n, 1.0f, 0), m->esz, kBpttHeader).total;
  return RLT_OK;
}

int rlt_bptt(const rlt_model* m, const void* e, const void* mem, int32_t T_mem, int32_t B, int32_t n,
             const int32_t* actions, float temperature, int32_t top_k, int32_t detach_s_every, int32_t flags,
             float* loss, float* logp, const rlt_grads* grads, float* d_e, float* d_mem, void* ws, size_t ws_bytes,
             rlt_stream_t stream) {
  if (!m || !e || !mem || !actions || !loss || !grads || !ws) return RLT_EINVAL;
  if (B <= 0 || n <= 0 || T_mem < n) return RLT_EINVAL;
  if (!(temperature > 0.f) || top_k < 0 || detach_s_every < 0) return RLT_EINVAL;
  if (flags & ~(RLT_DETACH_CACHE | RLT_DETACH_MEMORY | RLT_BPTT_NO_GRAPHS | RLT_BPTT_CORE_MEMGRAD)) return RLT_EINVAL;
  const float* gp[] = {grads->W_g, grads->b_g, grads->W_qkv, grads->W_O, grads->W_Qx, grads->W_Ox, grads->W_1,
                       grads->W_3, grads->W_2, grads->W_o, grads->dec_attn_norm, grads->dec_xattn_norm,
                       grads->dec_ffn_norm, grads->head_norm, grads->s_star};
  for (const float* p : gp)
    if (!p || !aligned16(p)) return RLT_EINVAL;
  if (!aligned16(e) || !aligned16(mem) || !aligned16(ws) || !aligned16(actions) || (d_e && !aligned16(d_e)) ||
      (d_mem && !aligned16(d_mem)) || (logp && !aligned16(logp)))
    return RLT_EINVAL;
  // bf16 models: d logits [B][V] and W_o^T [d][V] are tensor-core operands
  // with a row pitch of V elements (16-byte multiples)
  if (m->cfg.dtype == RLT_BF16 && m->cfg.vocab % 8 != 0) return RLT_EUNSUPPORTED;
  // the memory-gradient grid has one row per (sequence, head)
  if ((int64_t)B * m->cfg.n_heads > 65535) return RLT_EUNSUPPORTED;
  const bpplan::Shape S = bptt_shape(m, B, n, T_mem, temperature, top_k);
  if (ws_bytes < bpplan::layout(S, m->esz, kBpttHeader).total) return RLT_EWORKSPACE;
  int rc = bptt_attrs();
  if (rc) return rc;
  bpplan::Detach D;
  D.s_every = detach_s_every;
  D.cache = (flags & RLT_DETACH_CACHE) != 0;
  D.memory = (flags & RLT_DETACH_MEMORY) != 0;
  const bool graphs = (flags & RLT_BPTT_NO_GRAPHS) == 0;
  const bool mg_tc = (flags & RLT_BPTT_CORE_MEMGRAD) == 0;
  bpplan::Grads G;
  G.W_g = grads->W_g;
  G.b_g = grads->b_g;
  G.W_qkv = grads->W_qkv;
  G.W_O = grads->W_O;
  G.W_Qx = grads->W_Qx;
  G.W_Ox = grads->W_Ox;
  G.W_1 = grads->W_1;
  G.W_3 = grads->W_3;
  G.W_2 = grads->W_2;
  G.W_o = grads->W_o;
  G.attn_norm = grads->dec_attn_norm;
  G.xattn_norm = grads->dec_xattn_norm;
  G.ffn_norm = grads->dec_ffn_norm;
  G.head_norm = grads->head_norm;
  G.s_star = grads->s_star;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (m->cfg.dtype == RLT_BF16) {
    bpplan::Io<bf16> io{static_cast<const bf16*>(e), static_cast<const bf16*>(mem), actions, loss, logp, d_e, d_mem};
    return bptt_impl<bf16>(m, S, D, io, G, ws, s, graphs, mg_tc);
  }
  bpplan::Io<float> io{static_cast<const float*>(e), static_cast<const float*>(mem), actions, loss, logp, d_e, d_mem};
  return bptt_impl<float>(m, S, D, io, G, ws, s, graphs, mg_tc);
}

}  // extern "C"
