// cp_host.cu -- the C ABI: handle creation (validation, residency, weight
// repacking, scratch, schedule), frame launches, status and test hooks.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "cp.h"
#include "cp_internal.h"

namespace cp {
// Two builds of cp_kernel.cu: `generic` reads every size from the kernel
// parameters; `cp17` has the CodePredictor-1.7B sizes fixed (kShape1p7b).
namespace generic {
const void* frame_kernel_fn();
cudaError_t launch_frame(const KParams& prm, int grid, int cluster, int smem, cudaStream_t stream, bool pdl);
cudaError_t launch_test_philox(const uint32_t* ctr, const uint32_t* key, int n, int use_curand, uint32_t* out,
                               cudaStream_t s);
cudaError_t launch_test_draw(const float* logits, int rows, int V, const float* temp, const int32_t* topk,
                             const float* topp, const uint64_t* seed, const int64_t* offset, int group,
                             int32_t* codes, cudaStream_t s);
}  // namespace generic
namespace cp17 {
const void* frame_kernel_fn();
cudaError_t launch_frame(const KParams& prm, int grid, int cluster, int smem, cudaStream_t stream, bool pdl);
}  // namespace cp17
namespace cp17r128 {  // the same sizes, handles of more than 64 rows (M = 128 projections)
const void* frame_kernel_fn();
cudaError_t launch_frame(const KParams& prm, int grid, int cluster, int smem, cudaStream_t stream, bool pdl);
}  // namespace cp17r128
}  // namespace cp

using namespace cp;

struct cp_handle {
  int device = 0;
  Shape s{};
  int max_rows = 0;
  int C = 4, G = 0, smem = 0, sm_count = 0;
  bool fixed = false;      // runs the build specialised for kShape1p7b
  Plan* plan = nullptr;
  PlanView pv{};
  KParams base{};          // pointers and shape; per-frame fields filled at launch
  std::vector<void*> allocs;
  FrameArgs* d_fa = nullptr;
  float* d_embsum = nullptr;
  int64_t scratch_bytes = 0;
  std::vector<int> cuts;
  cudaStream_t cap_stream = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t graph_exec = nullptr;
  int last_rows = 0;
};

namespace {

// The frame kernel build a handle runs: the one with its shape fixed at
// compile time when the handle's shape and cluster are kShape1p7b.
bool matches_1p7b(const Shape& s, int C) {
  const FixedShape& f = kShape1p7b;
  return s.L == f.L && s.H == f.H && s.Hq == f.Hq && s.Hkv == f.Hkv && s.D == f.D && s.F == f.F && s.P == f.P &&
         s.V == f.V && s.T == f.T && s.qk_norm == f.qk_norm && C == f.cluster;
}
const void* frame_fn(const cp_handle* h) {
  if (!h->fixed) return generic::frame_kernel_fn();
  return h->s.MR > kRowsM64 ? cp17r128::frame_kernel_fn() : cp17::frame_kernel_fn();
}
cudaError_t launch(const cp_handle* h, const KParams& prm, cudaStream_t stream, bool pdl) {
  if (!h->fixed) return generic::launch_frame(prm, h->G, h->C, h->smem, stream, pdl);
  return h->s.MR > kRowsM64 ? cp17r128::launch_frame(prm, h->G, h->C, h->smem, stream, pdl)
                            : cp17::launch_frame(prm, h->G, h->C, h->smem, stream, pdl);
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

int to_shape(const cp_shape* in, Shape* s) {
  s->L = in->layers; s->H = in->hidden; s->Hq = in->q_heads; s->Hkv = in->kv_heads; s->D = in->head_dim;
  s->F = in->ffn; s->P = in->positions; s->V = in->vocab; s->T = in->talker_hidden;
  s->MR = in->max_rows > kRowsM64 ? kMaxRows : kRowsM64;  // row stride of the frame's buffers
  s->eps = in->rms_eps; s->rope_base = in->rope_base; s->qk_norm = in->qk_norm;
  return CP_OK;
}

// Limits of the kernels (documented in cp.h).
int check_shape(const cp_shape* in, int C) {
  if (!in) return CP_ERR_INVALID_ARG;
  const int L = in->layers, H = in->hidden, Hq = in->q_heads, Hkv = in->kv_heads, D = in->head_dim;
  const int F = in->ffn, P = in->positions, V = in->vocab, T = in->talker_hidden;
  if (L < 1 || H < 1 || Hq < 1 || Hkv < 1 || D < 1 || F < 1 || P < 1 || V < 1 || T < 1) return CP_ERR_INVALID_ARG;
  if (in->max_rows < 1 || in->max_rows > kMaxRows) return CP_ERR_UNSUPPORTED;
  if (!(in->rms_eps >= 0.f) || !(in->rope_base > 0.f)) return CP_ERR_INVALID_ARG;
  if (C != 2 && C != 4 && C != 8) return CP_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return CP_ERR_UNSUPPORTED;
  if (Hq % Hkv || Hkv > 16 || (Hq / Hkv != 1 && Hq / Hkv != 2 && Hq / Hkv != 4)) return CP_ERR_UNSUPPORTED;
  if (P < 2 || P > kMaxPositions) return CP_ERR_UNSUPPORTED;
  if (V % 256 || V > kMaxVocab) return CP_ERR_UNSUPPORTED;
  if (H % (64 * C) || (Hq * D) % (64 * C) || F % (64 * C) || T % (64 * C) || F % 64) return CP_ERR_UNSUPPORTED;
  if (H / 32 % 4 || H > 2048) return CP_ERR_UNSUPPORTED;  // the row scale reads up to 16 x 4 sums
  // per-chunk dependency counters: one per gate/up tile must fit a phase's counters
  if ((F % 96 == 0 ? F / 96 : F / 64) > kCounterStride) return CP_ERR_UNSUPPORTED;
  return CP_OK;
}

int cuda_err(cudaError_t e) { return e == cudaSuccess ? CP_OK : CP_ERR_CUDA; }

template <class T>
int dalloc(cp_handle* h, T** p, size_t bytes, bool zero = true) {
  void* v = nullptr;
  if (cudaMalloc(&v, bytes ? bytes : 16) != cudaSuccess) return CP_ERR_NOMEM;
  h->allocs.push_back(v);
  if (zero && cudaMemset(v, 0, bytes ? bytes : 16) != cudaSuccess) return CP_ERR_CUDA;
  *p = static_cast<T*>(v);
  h->scratch_bytes += (int64_t)bytes;
  return CP_OK;
}

// Copy `bytes` from a host or device pointer into host memory.
int fetch(void* dst, const void* src, size_t bytes) {
  if (!src) return CP_ERR_INVALID_ARG;
  return cudaMemcpy(dst, src, bytes, cudaMemcpyDefault) == cudaSuccess ? CP_OK : CP_ERR_INVALID_ARG;
}

// Pack one projection's tile grid: tile t, K part r, chunk kc, tile row f,
// 16-byte unit u -> base + ((t*C + r)*nkc + kc)*F*128 + f*128 + (u ^ (f&7))*16.
// `row_of(t, f)` names the source row ([out][in], width K) of tile row f.
template <class RowOf>
void pack_grid(uint8_t* dst, const Shape& s, int kind, int C, RowOf row_of) {
  const int F = proj_nfeat(s, kind), K = proj_k(s, kind), nt = proj_ntiles(s, kind);
  const int Ks = K / C, nkc = Ks / 64;
  for (int t = 0; t < nt; ++t)
    for (int r = 0; r < C; ++r)
      for (int kc = 0; kc < nkc; ++kc) {
        uint8_t* chunk = dst + (((size_t)t * C + r) * nkc + kc) * (size_t)F * 128;
        for (int f = 0; f < F; ++f) {
          const uint16_t* src = row_of(t, f) + (size_t)r * Ks + (size_t)kc * 64;
          for (int u = 0; u < 8; ++u) std::memcpy(chunk + (size_t)f * 128 + ((u ^ (f & 7)) * 16), src + u * 8, 16);
        }
      }
}

}  // namespace

extern "C" {

const char* cp_strerror(int st) {
  switch (st) {
    case CP_OK: return "ok";
    case CP_ERR_INVALID_ARG: return "invalid argument";
    case CP_ERR_UNSUPPORTED: return "unsupported shape, row count or device";
    case CP_ERR_RESIDENCY: return "the frame's CTAs cannot all be resident on this device";
    case CP_ERR_CUDA: return "CUDA runtime error";
    case CP_ERR_TIMEOUT: return "a device-side wait timed out";
    case CP_ERR_DEVICE_BOUNDS: return "an index outside its range reached the device";
    case CP_ERR_NOMEM: return "out of memory";
    case CP_ERR_PLAN: return "the static schedule failed validation";
    case CP_ERR_SCRATCH_LIMIT: return "the frame's working set does not fit the static scratch array";
    case CP_ERR_RANGE: return "a normed projection's partial sum left the fp16 range of its exchange";
  }
  return "unknown status";
}

void cp_destroy(cp_handle* h) {
  if (!h) return;
  {
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    if (h->graph_exec) cudaGraphExecDestroy(h->graph_exec);
    if (h->graph) cudaGraphDestroy(h->graph);
    if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
    for (void* p : h->allocs) cudaFree(p);
  }
  if (h->plan) plan_free(h->plan);
  delete h;
}

int cp_plan_check(const cp_shape* shape, int grid, int cluster, int chunk_waits, int corrupt, cp_plan_stats* out) {
  int st = check_shape(shape, cluster);
  if (out) std::memset(out, 0, sizeof(*out));
  if (st != CP_OK) {
    if (out) std::snprintf(out->message, sizeof(out->message), "%s", cp_strerror(st));
    return st;
  }
  Shape s;
  to_shape(shape, &s);
  Plan* p = nullptr;
  char msg[160] = {0};
  if (plan_build(s, grid, cluster, chunk_waits != 0, &p, msg, sizeof msg)) {
    if (out) std::snprintf(out->message, sizeof(out->message), "%s", msg);
    return CP_ERR_PLAN;
  }
  const int bad = plan_check(p, corrupt, msg, sizeof msg);
  if (out) {
    PlanView v = plan_view(p);
    out->phases = v.nph; out->tasks = v.ntasks; out->counters = v.ncounters;
    out->weight_bytes = v.weight_bytes; out->max_cta_weight_bytes = v.max_cta_bytes;
    out->min_cta_weight_bytes = v.min_cta_bytes; out->max_tasks_per_cta = v.max_tasks_per_cta;
    std::snprintf(out->message, sizeof(out->message), "%s", msg);
  }
  plan_free(p);
  return bad ? CP_ERR_PLAN : CP_OK;
}

int cp_create(const cp_shape* shape, const cp_weights* w, int device, const cp_options* opt, cp_handle** out) {
  if (!out || !shape || !w) return CP_ERR_INVALID_ARG;
  *out = nullptr;
  const int C = (opt && opt->cluster) ? opt->cluster : 4;
  int st = check_shape(shape, C);
  if (st != CP_OK) return st;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return CP_ERR_UNSUPPORTED;
  DeviceGuard guard(device);
  cudaDeviceProp prop{};
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return CP_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return CP_ERR_UNSUPPORTED;  // the binary is sm_103a only

  cp_handle* h = new (std::nothrow) cp_handle();
  if (!h) return CP_ERR_NOMEM;
  h->device = device;
  h->C = C;
  h->max_rows = shape->max_rows;
  to_shape(shape, &h->s);
  const Shape& s = h->s;
  h->fixed = !(opt && opt->generic_kernel) && matches_1p7b(s, C);
  h->sm_count = prop.multiProcessorCount;
  h->smem = kSmemBytes;
  auto fail = [&](int code) {
    cp_destroy(h);
    return code;
  };

  // Residency: every CTA of the persistent launch must be resident at once.
  const void* fn = frame_fn(h);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, h->smem) != cudaSuccess)
    return fail(CP_ERR_CUDA);
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((h->sm_count / C) * C);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = h->smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int ncl = 0;
    if (cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg) != cudaSuccess) return fail(CP_ERR_CUDA);
    int G = std::min(ncl, h->sm_count / C) * C;
    if (opt && opt->max_ctas > 0) G = std::min(G, (opt->max_ctas / C) * C);
    if (G < 2 * C) return fail(CP_ERR_RESIDENCY);
    h->G = G;
  }

  // Schedule.
  {
    char msg[160] = {0};
    if (plan_build(s, h->G, C, !(opt && opt->phase_waits), &h->plan, msg, sizeof msg)) return fail(CP_ERR_PLAN);
    if (plan_check(h->plan, 0, msg, sizeof msg)) {
      std::fprintf(stderr, "cp_create: schedule check failed: %s\n", msg);
      return fail(CP_ERR_PLAN);
    }
    h->pv = plan_view(h->plan);
  }
  const PlanView& pv = h->pv;

  // Weights: fetch to host, repack, upload.
  KParams& k = h->base;
  const int L = s.L, H = s.H, Hq = s.Hq, Hkv = s.Hkv, D = s.D, F = s.F, P = s.P, V = s.V, T = s.T;
  {
    std::vector<uint8_t> pack((size_t)pv.wpack_bytes);
    std::vector<uint16_t> a, b2;
    auto grab = [&](std::vector<uint16_t>& buf, const void* src, size_t n) {
      buf.resize(n);
      return fetch(buf.data(), src, n * 2);
    };
    // Offsets in the same order as the scheduler lays them out.
    size_t off = 0;
    auto grid_bytes = [&](int kind) {
      return (size_t)proj_ntiles(s, kind) * proj_nfeat(s, kind) * proj_k(s, kind) * 2;
    };
    if (grab(a, w->in_proj, (size_t)H * T)) return fail(CP_ERR_INVALID_ARG);
    pack_grid(pack.data() + off, s, K_INPROJ, C, [&](int t, int f) { return a.data() + (size_t)(t * 32 + f) * T; });
    off += grid_bytes(K_INPROJ);
    const int grp = Hq / Hkv;
    for (int l = 0; l < L; ++l) {
      if (!w->w_qkv || grab(a, w->w_qkv[l], (size_t)(Hq + 2 * Hkv) * D * H)) return fail(CP_ERR_INVALID_ARG);
      pack_grid(pack.data() + off, s, K_QKV, C, [&](int t, int f) {
        const int g = t / (grp + 2), wv = t % (grp + 2);
        size_t r;
        if (wv < grp) r = (size_t)(g * grp + wv) * D + f;
        else if (wv == grp) r = (size_t)Hq * D + (size_t)g * D + f;
        else r = (size_t)(Hq + Hkv) * D + (size_t)g * D + f;
        return a.data() + r * H;
      });
      off += grid_bytes(K_QKV);
      if (!w->w_o || grab(a, w->w_o[l], (size_t)H * Hq * D)) return fail(CP_ERR_INVALID_ARG);
      pack_grid(pack.data() + off, s, K_O, C, [&](int t, int f) { return a.data() + (size_t)(t * 32 + f) * Hq * D; });
      off += grid_bytes(K_O);
      if (!w->w_gate || !w->w_up || grab(a, w->w_gate[l], (size_t)F * H) || grab(b2, w->w_up[l], (size_t)F * H))
        return fail(CP_ERR_INVALID_ARG);
      pack_grid(pack.data() + off, s, K_GU, C, [&](int t, int f) {
        const size_t r = (size_t)t * (proj_nfeat(s, K_GU) / 2) + f / 2;
        return (f & 1 ? b2.data() : a.data()) + r * H;
      });
      off += grid_bytes(K_GU);
      if (!w->w_down || grab(a, w->w_down[l], (size_t)H * F)) return fail(CP_ERR_INVALID_ARG);
      pack_grid(pack.data() + off, s, K_DOWN, C, [&](int t, int f) { return a.data() + (size_t)(t * 32 + f) * F; });
      off += grid_bytes(K_DOWN);
    }
    for (int j = 0; j < P - 1; ++j) {
      if (!w->heads || grab(a, w->heads[j], (size_t)V * H)) return fail(CP_ERR_INVALID_ARG);
      pack_grid(pack.data() + off, s, K_HEAD, C, [&](int t, int f) { return a.data() + (size_t)(t * 64 + f) * H; });
      off += grid_bytes(K_HEAD);
    }
    if ((int64_t)off != pv.wpack_bytes) return fail(CP_ERR_PLAN);
    uint8_t* d;
    if ((st = dalloc(h, &d, off, false))) return fail(st);
    if (cudaMemcpy(d, pack.data(), off, cudaMemcpyHostToDevice) != cudaSuccess) return fail(CP_ERR_CUDA);
    k.wpack = d;
  }
  {
    // Embedding tables, norm gains, RoPE table.
    std::vector<uint16_t> buf;
    auto upload_list = [&](const void* const* list, int n, size_t each, uint16_t** dst) -> int {
      if (!list) return CP_ERR_INVALID_ARG;
      buf.resize(each * n);
      for (int i = 0; i < n; ++i)
        if (fetch(buf.data() + each * i, list[i], each * 2)) return CP_ERR_INVALID_ARG;
      int e = dalloc(h, dst, each * n * 2, false);
      if (e) return e;
      return cudaMemcpy(*dst, buf.data(), each * n * 2, cudaMemcpyHostToDevice) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
    };
    uint16_t* d;
    if ((st = upload_list(w->embed, P, (size_t)V * H, &d))) return fail(st);
    k.embed = d;
    if ((st = upload_list(w->attn_norm, L, H, &d))) return fail(st);
    k.attn_norm = d;
    if ((st = upload_list(w->mlp_norm, L, H, &d))) return fail(st);
    k.mlp_norm = d;
    if (s.qk_norm) {
      if ((st = upload_list(w->q_norm, L, D, &d))) return fail(st);
      k.q_norm = d;
      if ((st = upload_list(w->k_norm, L, D, &d))) return fail(st);
      k.k_norm = d;
    }
    const void* fn1[1] = {w->final_norm};
    if ((st = upload_list(fn1, 1, H, &d))) return fail(st);
    k.final_norm = d;
    std::vector<float> rope((size_t)P * (D / 2) * 2);
    for (int p = 0; p < P; ++p)
      for (int i = 0; i < D / 2; ++i) {
        const double ang = (double)p * std::pow((double)s.rope_base, -2.0 * i / D);
        rope[((size_t)p * (D / 2) + i) * 2] = (float)std::cos(ang);
        rope[((size_t)p * (D / 2) + i) * 2 + 1] = (float)std::sin(ang);
      }
    float* dr;
    if ((st = dalloc(h, &dr, rope.size() * 4, false))) return fail(st);
    if (cudaMemcpy(dr, rope.data(), rope.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess) return fail(CP_ERR_CUDA);
    k.rope = dr;
  }
  // Scratch.
  {
    const size_t MR = (size_t)s.MR;
    if ((st = dalloc(h, &k.x, (size_t)P * MR * H * 4))) return fail(st);
    if ((st = dalloc(h, &k.ssq, (size_t)P * MR * (H / 32) * 4))) return fail(st);
    if ((st = dalloc(h, &k.q, MR * Hq * D * 2))) return fail(st);
    if ((st = dalloc(h, &k.kv, (size_t)L * Hkv * ((MR + 7) / 8) * P * 8 * 2 * D * 2))) return fail(st);
    if ((st = dalloc(h, &k.o, MR * Hq * D * 2))) return fail(st);
    if ((st = dalloc(h, &k.m, MR * (size_t)F * 2))) return fail(st);
    if ((st = dalloc(h, &k.xb, (size_t)P * MR * H * 2))) return fail(st);
    if ((st = dalloc(h, &k.logits, (size_t)(P - 1) * MR * V * 4))) return fail(st);
    if ((st = dalloc(h, &h->d_embsum, MR * (size_t)H * 4))) return fail(st);
    if ((st = dalloc(h, &k.counters, (size_t)pv.ncounters * 4))) return fail(st);
    if ((st = dalloc(h, &k.status, 8 * 4))) return fail(st);
    if ((st = dalloc(h, &h->d_fa, sizeof(FrameArgs)))) return fail(st);
    const bool trace = opt && opt->trace;
    if (trace && (st = dalloc(h, &k.trace, (size_t)pv.ntasks * kTraceStamps * 8))) return fail(st);
    Task* dt;
    int32_t* di;
    if ((st = dalloc(h, &dt, (size_t)pv.ntasks * sizeof(Task), false))) return fail(st);
    if (cudaMemcpy(dt, pv.tasks, (size_t)pv.ntasks * sizeof(Task), cudaMemcpyHostToDevice)) return fail(CP_ERR_CUDA);
    k.tasks = dt;
    if ((st = dalloc(h, &di, (size_t)(pv.grid + 1) * 4, false))) return fail(st);
    if (cudaMemcpy(di, pv.task_start, (size_t)(pv.grid + 1) * 4, cudaMemcpyHostToDevice)) return fail(CP_ERR_CUDA);
    k.task_start = di;
    if ((st = dalloc(h, &di, (size_t)pv.grid * (pv.nph + 1) * 4, false))) return fail(st);
    if (cudaMemcpy(di, pv.phase_start, (size_t)pv.grid * (pv.nph + 1) * 4, cudaMemcpyHostToDevice))
      return fail(CP_ERR_CUDA);
    k.phase_start = di;
  }
  k.fa_dev = h->d_fa;
  k.s = s;
  k.attn_scale = (float)(1.0 / std::sqrt((double)D));
  k.cluster = C;
  k.m128 = s.MR > kRowsM64 ? 1 : 0;
  k.nph = pv.nph;
  k.ncounters = pv.ncounters;
  k.timeout_ns = (opt && opt->timeout_ns > 0) ? opt->timeout_ns : 2000000000LL;
  k.stall_task = (opt && opt->debug_stall_task > 0) ? pv.task_start[0] + opt->debug_stall_task - 1 : -1;
  k.stall_staging = (opt && opt->debug_stall_staging) ? 1 : 0;
  if (opt && opt->n_cuts > 0) {
    if (!opt->cuts) return fail(CP_ERR_INVALID_ARG);
    int prev = 0;
    for (int i = 0; i < opt->n_cuts; ++i) {
      if (opt->cuts[i] <= prev || opt->cuts[i] >= pv.nph) return fail(CP_ERR_INVALID_ARG);
      prev = opt->cuts[i];
      h->cuts.push_back(prev);
    }
  }
  if (cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking) != cudaSuccess) return fail(CP_ERR_CUDA);
  if (cudaDeviceSynchronize() != cudaSuccess) return fail(CP_ERR_CUDA);
  *out = h;
  return CP_OK;
}

static int fill_args(cp_handle* h, const float* hid, const int32_t* c0, const cp_sampler* sp, int rows,
                     int32_t* codes, float* emb_sum, FrameArgs* fa) {
  if (!h || !hid || !c0 || !sp || !codes) return CP_ERR_INVALID_ARG;
  if (!sp->temperature || !sp->top_k || !sp->top_p || !sp->seed || !sp->offset) return CP_ERR_INVALID_ARG;
  if (rows < 1 || rows > h->max_rows) return CP_ERR_INVALID_ARG;
  fa->h = hid; fa->c0 = c0; fa->temperature = sp->temperature; fa->top_k = sp->top_k; fa->top_p = sp->top_p;
  fa->seed = sp->seed; fa->offset = sp->offset; fa->codes = codes;
  fa->emb_sum = emb_sum ? emb_sum : h->d_embsum;
  fa->write_emb_sum = emb_sum != nullptr;
  fa->rows = rows;
  return CP_OK;
}

int cp_frame(cp_handle* h, const float* hid, const int32_t* c0, const cp_sampler* sp, int rows, int32_t* codes,
             float* emb_sum, cp_stream_t stream) {
  FrameArgs fa{};
  int st = fill_args(h, hid, c0, sp, rows, codes, emb_sum, &fa);
  if (st) return st;
  DeviceGuard g(h->device);
  KParams prm = h->base;
  prm.fa = fa;
  prm.mode = 0;
  std::vector<int> b;
  b.push_back(0);
  for (int c : h->cuts) b.push_back(c);
  b.push_back(h->pv.nph);
  for (size_t i = 0; i + 1 < b.size(); ++i) {
    prm.phase_lo = b[i];
    prm.phase_hi = b[i + 1];
    prm.last_launch = i + 2 == b.size();
    if (launch(h, prm, reinterpret_cast<cudaStream_t>(stream), false) != cudaSuccess)
      return CP_ERR_CUDA;
  }
  h->last_rows = rows;
  return CP_OK;
}

// ------------------------------------------------------------ static scratch
// The working set of cp_frame_static. In host code this name is a host-side
// stand-in, not a device address: kernels get the address that
// cudaGetSymbolAddress returns for the current device, looked up once per
// device (std::call_once: two host threads making their first call together
// look it up once).
static __device__ __align__(256) unsigned char g_frame_scratch[CP_STATIC_SCRATCH_BYTES];
constexpr int kMaxDevices = 128;
static std::once_flag g_scratch_once[kMaxDevices];
static void* g_scratch_addr[kMaxDevices];
static cudaError_t g_scratch_err[kMaxDevices];

int cp_frame_static(cp_handle* h, const float* hid, const int32_t* c0, const cp_sampler* sp, int rows,
                    int32_t* codes, float* emb_sum, cp_stream_t stream) {
  FrameArgs fa{};
  int st = fill_args(h, hid, c0, sp, rows, codes, emb_sum, &fa);
  if (st) return st;
  const Shape& s = h->s;
  // Carve the working set with a row stride of `rows`; every region 256-B aligned.
  // The status words stay in the handle (cp_status reads them, and a sticky
  // error skips this call as it skips cp_frame).
  const size_t R = (size_t)rows;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  };
  const size_t o_x = take((size_t)s.P * R * s.H * 4);
  const size_t o_ssq = take((size_t)s.P * R * (s.H / 32) * 4);
  const size_t o_q = take(R * s.Hq * s.D * 2);
  const size_t o_kv = take((size_t)s.L * s.Hkv * ((R + 7) / 8) * s.P * 8 * 2 * s.D * 2);
  const size_t o_o = take(R * s.Hq * s.D * 2);
  const size_t o_m = take(R * (size_t)s.F * 2);
  const size_t o_xb = take((size_t)s.P * R * s.H * 2);
  const size_t o_lg = take((size_t)(s.P - 1) * R * s.V * 4);
  const size_t o_es = take(R * (size_t)s.H * 4);
  const size_t o_cnt = take((size_t)h->pv.ncounters * 4);
  if (off > CP_STATIC_SCRATCH_BYTES) return CP_ERR_SCRATCH_LIMIT;
  if (h->device < 0 || h->device >= kMaxDevices) return CP_ERR_UNSUPPORTED;
  DeviceGuard g(h->device);
  std::call_once(g_scratch_once[h->device], [&] {
    void* ptr = nullptr;
    g_scratch_err[h->device] = cudaGetSymbolAddress(&ptr, g_frame_scratch);
    g_scratch_addr[h->device] = ptr;
  });
  if (g_scratch_err[h->device] != cudaSuccess || !g_scratch_addr[h->device]) return CP_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(g_scratch_addr[h->device]);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // The counters must start at zero (the last call's contents stay in the
  // array); everything else is written before it is read.
  if (cudaMemsetAsync(base + o_cnt, 0, off - o_cnt, cs) != cudaSuccess) return CP_ERR_CUDA;
  KParams prm = h->base;
  prm.x = reinterpret_cast<float*>(base + o_x);
  prm.ssq = reinterpret_cast<float*>(base + o_ssq);
  prm.q = reinterpret_cast<uint16_t*>(base + o_q);
  prm.kv = reinterpret_cast<uint16_t*>(base + o_kv);
  prm.o = reinterpret_cast<uint16_t*>(base + o_o);
  prm.m = reinterpret_cast<uint16_t*>(base + o_m);
  prm.xb = reinterpret_cast<uint16_t*>(base + o_xb);
  prm.logits = reinterpret_cast<float*>(base + o_lg);
  prm.counters = reinterpret_cast<uint32_t*>(base + o_cnt);
  prm.trace = nullptr;
  prm.s.MR = rows;
  if (!emb_sum) fa.emb_sum = reinterpret_cast<float*>(base + o_es);
  prm.fa = fa;
  prm.mode = 0;
  prm.phase_lo = 0;
  prm.phase_hi = h->pv.nph;
  prm.last_launch = 1;
  return launch(h, prm, cs, false) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

int cp_frame_split(cp_handle* h, const float* hid, const int32_t* c0, const cp_sampler* sp, int rows,
                   int32_t* codes, float* emb_sum, cp_stream_t stream) {
  FrameArgs fa{};
  int st = fill_args(h, hid, c0, sp, rows, codes, emb_sum, &fa);
  if (st) return st;
  DeviceGuard g(h->device);
  if (!h->graph_exec) {
    KParams prm = h->base;
    prm.mode = 1;
    prm.last_launch = 0;
    if (cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return CP_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    for (int ph = 0; ph < h->pv.nph && e == cudaSuccess; ++ph) {
      prm.phase_lo = ph;
      prm.phase_hi = ph + 1;
      e = launch(h, prm, h->cap_stream, ph > 0);
    }
    cudaGraph_t graph = nullptr;
    const cudaError_t e2 = cudaStreamEndCapture(h->cap_stream, &graph);
    if (e != cudaSuccess || e2 != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      return CP_ERR_CUDA;
    }
    h->graph = graph;
    if (cudaGraphInstantiate(&h->graph_exec, graph, 0) != cudaSuccess) return CP_ERR_CUDA;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(h->d_fa, &fa, sizeof fa, cudaMemcpyHostToDevice, s) != cudaSuccess) return CP_ERR_CUDA;
  if (cudaGraphLaunch(h->graph_exec, s) != cudaSuccess) return CP_ERR_CUDA;
  h->last_rows = rows;
  return CP_OK;
}

int cp_debug_logits(cp_handle* h, int group, float* dst, cp_stream_t stream) {
  if (!h || !dst || group < 0 || group >= h->s.P - 1 || h->last_rows < 1) return CP_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  const size_t n = (size_t)h->last_rows * h->s.V;
  return cuda_err(cudaMemcpyAsync(dst, h->base.logits + (size_t)group * h->s.MR * h->s.V, n * 4,
                                  cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)));
}

int cp_debug_state(cp_handle* h, int what, int a, int b, void* dst, cp_stream_t stream) {
  if (!h || !dst || h->last_rows < 1) return CP_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  const Shape& s = h->s;
  const size_t R = (size_t)h->last_rows, MR = (size_t)s.MR;
  const void* src;
  size_t bytes;
  if (what == 0) {
    if (a < 0 || a >= s.P) return CP_ERR_INVALID_ARG;
    src = h->base.x + (size_t)a * MR * s.H;
    bytes = R * s.H * 4;
  } else if (what == 1 || what == 2) {
    // cache layout [L][Hkv][MR/8][P][8][key|value][D]: one 2-D copy per kv head and row block
    if (a < 0 || a >= s.L || b < 0 || b >= s.P) return CP_ERR_INVALID_ARG;
    const size_t D = s.D, RB = (MR + 7) / 8;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    for (size_t g = 0; g < (size_t)s.Hkv; ++g)
      for (size_t rb = 0; rb * 8 < R; ++rb) {
        const uint16_t* sp = h->base.kv + ((((size_t)a * s.Hkv + g) * RB + rb) * s.P + b) * 8 * 2 * D + (what == 2 ? D : 0);
        uint16_t* dp = static_cast<uint16_t*>(dst) + ((rb * 8) * s.Hkv + g) * D;
        const size_t nrow = std::min<size_t>(8, R - rb * 8);
        if (cudaMemcpy2DAsync(dp, (size_t)s.Hkv * D * 2, sp, 2 * D * 2, D * 2, nrow, cudaMemcpyDeviceToDevice, cs) !=
            cudaSuccess)
          return CP_ERR_CUDA;
      }
    return CP_OK;
  } else {
    return CP_ERR_INVALID_ARG;
  }
  return cuda_err(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)));
}

int cp_status(cp_handle* h) {
  if (!h) return CP_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  if (cudaDeviceSynchronize() != cudaSuccess) return CP_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, h->base.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return CP_ERR_CUDA;
  return v;
}

int cp_clear_status(cp_handle* h) {
  if (!h) return CP_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  if (cudaDeviceSynchronize() != cudaSuccess) return CP_ERR_CUDA;
  if (cudaMemset(h->base.status, 0, 8 * 4) != cudaSuccess) return CP_ERR_CUDA;
  if (cudaMemset(h->base.counters, 0, (size_t)h->pv.ncounters * 4) != cudaSuccess) return CP_ERR_CUDA;
  return cuda_err(cudaDeviceSynchronize());
}

int cp_get_info(const cp_handle* h, cp_info* out) {
  if (!h || !out) return CP_ERR_INVALID_ARG;
  out->grid = h->G;
  out->cluster = h->C;
  out->threads = kThreads;
  out->smem_bytes = h->smem;
  out->phases = h->pv.nph;
  out->tasks = h->pv.ntasks;
  out->weight_bytes = h->pv.weight_bytes;
  out->max_cta_weight_bytes = h->pv.max_cta_bytes;
  out->min_cta_weight_bytes = h->pv.min_cta_bytes;
  out->scratch_bytes = h->scratch_bytes;
  out->sm_count = h->sm_count;
  out->specialized = h->fixed ? 1 : 0;
  return CP_OK;
}

int cp_trace(cp_handle* h, int64_t* dst, cp_stream_t stream) {
  if (!h || !dst || !h->base.trace) return CP_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  return cuda_err(cudaMemcpyAsync(dst, h->base.trace, (size_t)h->pv.ntasks * kTraceStamps * 8,
                                  cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)));
}

int cp_test_philox(const uint32_t* ctr, const uint32_t* key, int n, int use_curand, uint32_t* out,
                   cp_stream_t stream) {
  if (!ctr || !key || !out || n < 1) return CP_ERR_INVALID_ARG;
  return cuda_err(generic::launch_test_philox(ctr, key, n, use_curand, out, reinterpret_cast<cudaStream_t>(stream)));
}

int cp_test_draw(const float* logits, int rows, int vocab, const cp_sampler* sp, int group, int32_t* codes,
                 cp_stream_t stream) {
  if (!logits || !sp || !codes || rows < 1 || vocab % 256 || vocab > kMaxVocab || vocab < 256)
    return CP_ERR_INVALID_ARG;
  if (!sp->temperature || !sp->top_k || !sp->top_p || !sp->seed || !sp->offset) return CP_ERR_INVALID_ARG;
  return cuda_err(generic::launch_test_draw(logits, rows, vocab, sp->temperature, sp->top_k, sp->top_p, sp->seed, sp->offset,
                                   group, codes, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
