// cp_plan.cpp -- the static per-CTA task schedule of one frame and its checker.
//
// "Qwen3-TTS: Run the 1.7B Depth Loop as One Persistent Kernel on Hopper",
// section "How it works": one launch walks a static task list per CTA built
// on the host; a task waits on a counter in global memory, runs one tile and
// signals a counter; an attention task waits only on the qkv tiles of its kv
// head; o and down split each tile's K loop across the CTAs of a cluster.
// "The gaps between kernels: PDL and megakernels", section "Megakernels":
// every CTA must be resident and a dependency may only point to an earlier
// instruction, so the earliest unfinished one can always run.
//
// Here every projection (input projection, qkv, o, gate/up, down, heads) is
// split along K over the C CTAs of a cluster; a tile is a cluster task whose
// C parts meet to add their partial sums in a fixed order.
#include "cp_internal.h"

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <map>
#include <new>
#include <string>
#include <vector>

namespace cp {

struct Plan {
  Shape s;
  int G = 0, C = 0, NC = 0;
  bool chunked = false;  // per-chunk waits (producers signal per chunk of their output)
  std::vector<Phase> phases;
  std::vector<std::vector<Task>> lists;
  std::vector<Task> flat;
  std::vector<int32_t> task_start;
  std::vector<int32_t> phase_start;
  std::vector<int32_t> counter_target;
  int64_t wpack_bytes = 0;
  int64_t weight_bytes = 0, max_cta = 0, min_cta = 0;
  int max_tasks = 0;
};

int proj_nfeat(const Shape& s, int kind) {
  switch (kind) {
    case K_INPROJ: return 32;
    case K_QKV: return s.D;
    case K_O: return 32;
    case K_GU: return s.F % 96 == 0 ? 192 : 128;  // gate and up rows interleaved: 96 (or 64) ffn features
    case K_DOWN: return 32;
    case K_HEAD: return 64;
  }
  return 0;
}

int proj_k(const Shape& s, int kind) {
  switch (kind) {
    case K_INPROJ: return s.T;
    case K_QKV: return s.H;
    case K_O: return s.Hq * s.D;
    case K_GU: return s.H;
    case K_DOWN: return s.F;
    case K_HEAD: return s.H;
  }
  return 0;
}

int proj_ntiles(const Shape& s, int kind) {
  switch (kind) {
    case K_INPROJ: return s.H / 32;
    case K_QKV: return s.Hq + 2 * s.Hkv;   // one head (D features) per tile, grouped by kv head
    case K_O: return s.H / 32;
    case K_GU: return 2 * s.F / proj_nfeat(s, K_GU);
    case K_DOWN: return s.H / 32;
    case K_HEAD: return s.V / 64;
  }
  return 0;
}

static void fmt(char* msg, int n, const std::string& m) {
  if (msg && n > 0) { std::snprintf(msg, n, "%s", m.c_str()); }
}

// Counter slot (within its phase's kCounterStride) that tile `tile` of a
// projection phase signals: the 64-feature chunk of x it wrote (input
// projection, o, down: tiles of 32 features), its own slot (gate/up), its kv
// group (qkv), one slot (heads).
static int tile_slot(const Shape& s, int kind, int tile, bool chunked) {
  if (!chunked) return kind == K_QKV ? tile / (s.Hq / s.Hkv + 2) : 0;  // one counter (qkv: per kv group)
  switch (kind) {
    case K_INPROJ: case K_O: case K_DOWN: return tile / 2;
    case K_GU: return tile;
    case K_QKV: return tile / (s.Hq / s.Hkv + 2);
    default: return 0;
  }
}
// Counter signalled by tile j (0 <= j < ntl) of a task.
static int tile_signal(const Shape&, const Task& t, int j) { return j == 0 ? t.signal : t.signal_b; }
static bool normed_kind(int kind) { return kind == K_QKV || kind == K_GU || kind == K_HEAD; }

// Every (counter, target) a task waits on before it completes: its single
// counters, the slots of each of its input chunks and, for a normed
// projection waiting per chunk of x, every chunk of x (the norm's row factor
// reads the whole row's sums of squares).
static std::vector<std::pair<int, int>> waits_of(const Shape& s, const Task& t) {
  std::vector<std::pair<int, int>> w;
  if (t.wait0 >= 0) w.push_back({t.wait0, t.target0});
  if (t.wait1 >= 0) w.push_back({t.wait1, t.target1});
  if (t.type == 1 /* T_PROJ */ && t.cbase >= 0) {
    const int fps = t.cpack >> 16, tg = t.cpack & 0xFFFF;
    for (int c = 0; c < t.nkc; ++c) {
      const int e0 = t.k0 + 64 * c;
      for (int sl = e0 / fps; sl <= (e0 + 63) / fps; ++sl) w.push_back({t.cbase + sl, tg});
    }
    if (normed_kind(t.kind))
      for (int sl = 0; sl < s.H / 64; ++sl) w.push_back({t.cbase + sl, tg});
  }
  return w;
}
static int task_tiles(const Task& t) { return t.type == T_PROJ ? t.ntl : 1; }

static bool is_proj(int kind) {
  return kind == K_INPROJ || kind == K_QKV || kind == K_O || kind == K_GU || kind == K_DOWN ||
         kind == K_HEAD;
}

int plan_build(const Shape& s, int G, int C, bool chunked, Plan** out, char* msg, int msglen) {
  *out = nullptr;
  if (C < 1 || G < C || G % C) { fmt(msg, msglen, "grid must be a positive multiple of the cluster"); return 1; }
  Plan* p = new (std::nothrow) Plan();
  if (!p) return 1;
  p->s = s; p->G = G; p->C = C; p->NC = G / C; p->chunked = chunked;
  const int grp = s.Hq / s.Hkv;
  const int nrb = s.MR / kRowBlock;

  // Packed weight layout: in_proj; per layer qkv, o, gate/up, down; heads.
  std::map<std::pair<int, int>, int64_t> wbase;
  int64_t off = 0;
  auto add = [&](int kind, int idx) {
    int F = proj_nfeat(s, kind), K = proj_k(s, kind), nt = proj_ntiles(s, kind);
    wbase[{kind, idx}] = off;
    off += (int64_t)nt * F * K * 2;
  };
  add(K_INPROJ, 0);
  for (int l = 0; l < s.L; ++l) { add(K_QKV, l); add(K_O, l); add(K_GU, l); add(K_DOWN, l); }
  for (int j = 0; j < s.P - 1; ++j) add(K_HEAD, j);
  p->wpack_bytes = off;

  // Phases in execution order.
  auto push = [&](int kind, int layer, int pos, int group) {
    Phase ph{};
    ph.kind = kind; ph.layer = layer; ph.pos = pos; ph.group = group;
    if (is_proj(kind)) {
      ph.ntiles = proj_ntiles(s, kind); ph.nfeat = proj_nfeat(s, kind); ph.K = proj_k(s, kind);
      ph.w_base = wbase[{kind, kind == K_HEAD ? group : (kind == K_INPROJ ? 0 : layer)}];
    }
    p->phases.push_back(ph);
  };
  push(K_INPROJ, -1, 0, -1);
  push(K_EMB0, -1, 1, 0);
  for (int pos = 0; pos < s.P; ++pos) {
    for (int l = 0; l < s.L; ++l) {
      push(K_QKV, l, pos, -1); push(K_ATTN, l, pos, -1); push(K_O, l, pos, -1);
      push(K_GU, l, pos, -1); push(K_DOWN, l, pos, -1);
    }
    if (pos >= 1) { push(K_HEAD, -1, pos, pos - 1); push(K_DRAW, -1, pos + 1, pos - 1); }
  }
  const int nph = (int)p->phases.size();
  auto find = [&](int kind, int layer, int pos) {
    for (int i = 0; i < nph; ++i) {
      const Phase& q = p->phases[i];
      if (q.kind == kind && q.layer == layer && q.pos == pos) return i;
    }
    return -1;
  };
  auto find_group = [&](int kind, int group) {
    for (int i = 0; i < nph; ++i)
      if (p->phases[i].kind == kind && p->phases[i].group == group) return i;
    return -1;
  };

  // Waits of each phase's tasks: single counters (wait0: the predecessor when
  // it signals one counter, or a kv group's; wait1: a second one) and the
  // per-chunk waits of a projection whose producer signals per chunk (slot
  // range of each 64-element input chunk: features per slot `fps`). Targets
  // are filled in once every task's signals are counted.
  struct Dep { int w0 = -1, w1 = -1, cph = -1, fps = 0; };
  std::vector<Dep> deps(nph);
  for (int i = 0; i < nph; ++i) {
    const Phase& q = p->phases[i];
    Dep& d = deps[i];
    // per-chunk waits, or (without them) one wait for the whole producer phase
    auto chunks = [&](int ph, int fps) {
      if (chunked) { d.cph = ph; d.fps = fps; }
      else d.w0 = ph * kCounterStride;
    };
    auto x_chunks = [&](int ph) { chunks(ph, 64); };
    switch (q.kind) {
      case K_QKV:
        if (q.layer > 0) x_chunks(find(K_DOWN, q.layer - 1, q.pos));
        else if (q.pos == 0) x_chunks(find(K_INPROJ, -1, 0));
        else if (q.pos == 1) {  // input from the first embedding; the earlier position's last
                                // layer must be done (buffers shared between positions)
          if (chunked) {
            d.w0 = find(K_EMB0, -1, 1) * kCounterStride;
            x_chunks(find(K_DOWN, s.L - 1, 0));
          } else {
            d.w0 = find(K_EMB0, -1, 1) * kCounterStride;
            d.w1 = find(K_DOWN, s.L - 1, 0) * kCounterStride;
          }
        } else d.w0 = find_group(K_DRAW, q.pos - 2) * kCounterStride;
        break;
      case K_O: chunks(find(K_ATTN, q.layer, q.pos), grp * s.D); break;
      case K_GU: x_chunks(find(K_O, q.layer, q.pos)); break;
      case K_DOWN: chunks(find(K_GU, q.layer, q.pos), proj_nfeat(s, K_GU) / 2); break;
      case K_HEAD: x_chunks(find(K_DOWN, s.L - 1, q.pos)); break;
      case K_DRAW: d.w0 = find_group(K_HEAD, q.group) * kCounterStride; break;
      default: break;
    }
  }

  p->lists.assign(G, {});
  int rot_cl = 0, rot_cta = 0;
  for (int i = 0; i < nph; ++i) {
    const Phase& q = p->phases[i];
    const Dep& d = deps[i];
    if (is_proj(q.kind)) {
      const int Ks = q.K / C, nkc = Ks / 64;
      const int cpp = std::max(1, std::min(nkc, kPageBytes / (q.nfeat * 128)));
      const int64_t unit = (int64_t)nkc * q.nfeat * 128;
      // Tiles per cluster task: one, or two adjacent tiles sharing the staged K part
      // when there are more tiles than clusters (up to twice as many) and the K part
      // fits the activation slots, so no cluster runs a second round.
      const int NC = p->NC;
      // (never for handles of more than 64 rows: their exchange has one receive slot)
      const int pairs = (s.MR <= kRowsM64 && q.ntiles > NC && q.ntiles <= 2 * NC && nkc <= kNumA) ? q.ntiles - NC
                                                                                                : 0;
      int t = 0, ci = 0;
      while (t < q.ntiles) {
        const int ntl = (ci < pairs) ? 2 : 1;
        const int cl = (rot_cl + ci) % NC;
        for (int r = 0; r < C; ++r) {
          Task k{};
          k.type = T_PROJ; k.kind = q.kind; k.layer = q.layer; k.pos = q.pos; k.group = q.group;
          k.tile = t; k.kslice = r; k.nfeat = q.nfeat; k.k0 = r * Ks; k.nkc = nkc; k.cpp = cpp;
          k.phase = i; k.wait0 = d.w0; k.wait1 = d.w1;
          k.cbase = d.cph >= 0 ? d.cph * kCounterStride : -1;
          k.cpack = d.fps << 16;
          k.signal = i * kCounterStride + tile_slot(s, q.kind, t, chunked);
          k.signal_b = ntl == 2 ? i * kCounterStride + tile_slot(s, q.kind, t + 1, chunked) : -1;
          k.ntl = ntl;
          k.w_off = q.w_base + ((int64_t)t * C + r) * unit;
          p->lists[cl * C + r].push_back(k);
        }
        t += ntl;
        ++ci;
      }
      rot_cl = (rot_cl + ci) % NC;
    } else {
      int n = q.kind == K_ATTN ? s.Hkv * nrb : s.MR;
      for (int u = 0; u < n; ++u) {
        Task k{};
        k.type = q.kind == K_ATTN ? T_ATTN : (q.kind == K_DRAW ? T_DRAW : T_EMB0);
        k.kind = q.kind; k.layer = q.layer; k.pos = q.pos; k.phase = i;
        k.group = q.kind == K_ATTN ? u / nrb : q.group;
        k.tile = q.kind == K_ATTN ? u % nrb : u;
        k.wait0 = d.w0; k.wait1 = -1; k.cbase = -1; k.cpack = 0; k.signal_b = -1;
        k.signal = i * kCounterStride;
        if (q.kind == K_ATTN) {
          // its kv group's qkv tiles; and the group's keys and values of the
          // earlier positions, copied before the task's own dependency is met
          k.wait0 = (i - 1) * kCounterStride + k.group;
          if (q.pos > 0) k.wait1 = find(K_QKV, q.layer, q.pos - 1) * kCounterStride + k.group;
          if (chunked) k.signal = i * kCounterStride + k.group;
        }
        k.ntl = 1;
        k.w_off = -1;
        p->lists[rot_cta % G].push_back(k);
        rot_cta = (rot_cta + 1) % G;
      }
    }
  }

  // Counter targets: the signals each counter gets; then every wait's target.
  p->counter_target.assign((size_t)nph * kCounterStride, 0);
  for (auto& L : p->lists)
    for (auto& t : L)
      for (int j = 0; j < task_tiles(t); ++j) p->counter_target[tile_signal(s, t, j)]++;
  for (auto& L : p->lists)
    for (auto& t : L) {
      t.target0 = t.wait0 >= 0 ? p->counter_target[t.wait0] : 0;
      t.target1 = t.wait1 >= 0 ? p->counter_target[t.wait1] : 0;
      if (t.cbase >= 0) {
        const int fps = t.cpack >> 16;
        t.cpack = (fps << 16) | p->counter_target[t.cbase + (t.k0 / fps)];
      }
    }

  // Flatten.
  p->task_start.assign(G + 1, 0);
  p->phase_start.assign((size_t)G * (nph + 1), 0);
  int64_t mx = 0, mn = INT64_MAX;
  for (int b = 0; b < G; ++b) {
    p->task_start[b] = (int32_t)p->flat.size();
    int64_t bytes = 0;
    int pi = 0;
    const auto& L = p->lists[b];
    for (size_t k = 0; k < L.size(); ++k) {
      while (pi <= L[k].phase) p->phase_start[(size_t)b * (nph + 1) + pi++] = (int32_t)p->flat.size();
      p->flat.push_back(L[k]);
      if (L[k].type == T_PROJ) bytes += (int64_t)L[k].ntl * L[k].nkc * L[k].nfeat * 128;
    }
    while (pi <= nph) p->phase_start[(size_t)b * (nph + 1) + pi++] = (int32_t)p->flat.size();
    p->weight_bytes += bytes;
    mx = std::max(mx, bytes); mn = std::min(mn, bytes);
    p->max_tasks = std::max(p->max_tasks, (int)L.size());
  }
  p->task_start[G] = (int32_t)p->flat.size();
  p->max_cta = mx; p->min_cta = mn;
  *out = p;
  return 0;
}

void plan_free(Plan* p) { delete p; }

PlanView plan_view(const Plan* p) {
  PlanView v{};
  v.tasks = p->flat.data(); v.ntasks = (int)p->flat.size();
  v.task_start = p->task_start.data(); v.grid = p->G;
  v.phase_start = p->phase_start.data(); v.nph = (int)p->phases.size();
  v.ncounters = (int)p->counter_target.size();
  v.wpack_bytes = p->wpack_bytes;
  v.weight_bytes = p->weight_bytes; v.max_cta_bytes = p->max_cta; v.min_cta_bytes = p->min_cta;
  v.max_tasks_per_cta = p->max_tasks;
  v.phases = p->phases.data();
  return v;
}

// ------------------------------------------------------------------ checker
int plan_check(const Plan* pin, int corrupt, char* msg, int msglen) {
  Plan p = *pin;  // copy: corruption for tests must not touch the real plan
  const int G = p.G, C = p.C, nph = (int)p.phases.size();
  const int NCt = (int)p.counter_target.size();
  auto& lists = p.lists;

  if (corrupt == 1) {          // a wait that asks for one signal more than its phase gives
    for (auto& L : lists) for (auto& t : L) {
      if (t.wait0 >= 0) { t.target0 += 1; goto done_corrupt; }
      if (t.cbase >= 0) { t.cpack += 1; goto done_corrupt; }
    }
  } else if (corrupt == 2) {   // a task moved ahead of the one it depends on
    for (auto& L : lists) {
      for (size_t k = 1; k < L.size(); ++k) {
        const auto w = waits_of(p.s, L[k]);
        for (size_t j = 0; j < k; ++j) {
          for (auto& cw : w)
            if (L[j].signal == cw.first) { std::swap(L[j], L[k]); goto done_corrupt; }
        }
      }
    }
  } else if (corrupt == 3) {   // two parts of one tile with the same rank
    for (auto& L : lists) for (auto& t : L) if (t.type == T_PROJ && t.kslice == 1) { t.kslice = 0; goto done_corrupt; }
  }
done_corrupt:

  // 1. signals per counter equal the wait targets; waits point to earlier phases.
  std::vector<int32_t> signals(NCt, 0);
  for (auto& L : lists) for (auto& t : L) {
    for (int j = 0; j < task_tiles(t); ++j) {
      const int sg = tile_signal(p.s, t, j);
      if (sg < 0 || sg >= NCt) { fmt(msg, msglen, "signal counter out of range"); return 1; }
      signals[sg]++;
    }
  }
  // each counter's signals against the count the phase structure gives in closed form
  {
    const int grp = p.s.Hq / p.s.Hkv, nrb = p.s.MR / kRowBlock;
    std::vector<int32_t> want(NCt, 0);
    for (int ph = 0; ph < nph; ++ph) {
      const Phase& q = p.phases[ph];
      int32_t* w = &want[(size_t)ph * kCounterStride];
      switch (q.kind) {
        case K_INPROJ: case K_O: case K_DOWN:
          if (p.chunked) for (int i = 0; i < q.ntiles / 2; ++i) w[i] = 2 * C;
          else w[0] = q.ntiles * C;
          break;
        case K_GU:
          if (p.chunked) for (int i = 0; i < q.ntiles; ++i) w[i] = C;
          else w[0] = q.ntiles * C;
          break;
        case K_QKV: for (int g = 0; g < p.s.Hkv; ++g) w[g] = (grp + 2) * C; break;
        case K_HEAD: w[0] = q.ntiles * C; break;
        case K_ATTN:
          if (p.chunked) for (int g = 0; g < p.s.Hkv; ++g) w[g] = nrb;
          else w[0] = p.s.Hkv * nrb;
          break;
        case K_DRAW: case K_EMB0: w[0] = p.s.MR; break;
        default: break;
      }
    }
    for (int c = 0; c < NCt; ++c) {
      if (signals[c] != want[c] || p.counter_target[c] != want[c]) {
        fmt(msg, msglen, "counter " + std::to_string(c) + " gets " + std::to_string(signals[c]) +
                             " signals, target " + std::to_string(p.counter_target[c]) + ", phase structure " +
                             std::to_string(want[c]));
        return 1;
      }
    }
  }
  for (int b = 0; b < G; ++b) {
    int last = -1;
    for (auto& t : lists[b]) {
      if (t.cbase >= 0 && (t.cbase % kCounterStride || t.type != T_PROJ || (t.cpack >> 16) < 1)) {
        fmt(msg, msglen, "per-chunk wait without a producer phase"); return 1;
      }
      for (auto& cw : waits_of(p.s, t)) {
        const int c = cw.first, tg = cw.second;
        if (c < 0 || c >= NCt) { fmt(msg, msglen, "wait counter out of range"); return 1; }
        if (c / kCounterStride >= t.phase) { fmt(msg, msglen, "task waits on its own or a later phase"); return 1; }
        if (tg != p.counter_target[c]) {
          fmt(msg, msglen, "wait target " + std::to_string(tg) + " on counter " + std::to_string(c) +
                               " differs from its " + std::to_string(p.counter_target[c]) + " signals");
          return 1;
        }
      }
      if (t.phase < last) { fmt(msg, msglen, "CTA " + std::to_string(b) + " list is not in phase order"); return 1; }
      last = t.phase;
      if (t.type == T_PROJ) {
        if (t.k0 + t.nkc * 64 > proj_k(p.s, t.kind)) { fmt(msg, msglen, "K part out of range"); return 1; }
        const int64_t unit = (int64_t)t.nkc * t.nfeat * 128;
        if (t.ntl < 1 || t.ntl > 2 || (t.ntl == 2 && (t.nkc > kNumA || p.s.MR > kRowsM64))) {
          fmt(msg, msglen, "tiles per task out of range"); return 1;
        }
        if (t.w_off < 0 || t.w_off + (int64_t)(t.ntl - 1) * C * unit + unit > p.wpack_bytes) {
          fmt(msg, msglen, "weight part out of the packed buffer"); return 1;
        }
        if (t.nfeat % 16 || t.nfeat < 16 || t.nfeat > kMaxTileN || t.nfeat * 128 > kPageBytes) {
          fmt(msg, msglen, "tile width not an MMA N that fits a page and an accumulator"); return 1;
        }
      }
    }
  }
  // 2. each K-split tile: C parts on one cluster, ranks 0..C-1 matching the CTA rank.
  std::map<std::pair<int, int>, std::vector<int>> parts;
  for (int b = 0; b < G; ++b)
    for (auto& t : lists[b])
      if (t.type == T_PROJ) {
        if (t.kslice != b % C) { fmt(msg, msglen, "tile part rank differs from its CTA's cluster rank"); return 1; }
        for (int j = 0; j < t.ntl; ++j) parts[{t.phase, t.tile + j}].push_back(b);
      }
  for (auto& kv : parts) {
    auto& v = kv.second;
    if ((int)v.size() != C) { fmt(msg, msglen, "tile with a wrong number of parts"); return 1; }
    std::sort(v.begin(), v.end());
    for (int r = 0; r < C; ++r)
      if (v[r] / C != v[0] / C || v[r] % C != r) { fmt(msg, msglen, "tile parts not on one cluster"); return 1; }
  }
  // 3. simulate: counters start at 0; a task runs when its waits hold; the C
  //    parts of a tile run together (they exchange partial sums).
  std::vector<int32_t> cnt(NCt, 0);
  std::vector<size_t> pc(G, 0);
  size_t remaining = 0;
  for (auto& L : lists) remaining += L.size();
  auto ready = [&](const Task& t) {
    for (auto& cw : waits_of(p.s, t))
      if (cnt[cw.first] < cw.second) return false;
    return true;
  };
  bool progress = true;
  while (remaining && progress) {
    progress = false;
    for (int b = 0; b < G; ++b) {
      while (pc[b] < lists[b].size()) {
        const Task& t = lists[b][pc[b]];
        if (!ready(t)) break;
        if (t.type == T_PROJ) {
          int base = (b / C) * C;
          bool all = true;
          for (int r = 0; r < C; ++r) {
            int c = base + r;
            if (pc[c] >= lists[c].size()) { all = false; break; }
            const Task& u = lists[c][pc[c]];
            // (each part waits for its own K part's chunks)
            if (u.type != T_PROJ || u.phase != t.phase || u.tile != t.tile || !ready(u)) { all = false; break; }
          }
          if (!all) break;
          for (int r = 0; r < C; ++r) {
            const Task& u = lists[base + r][pc[base + r]];
            if (u.ntl != t.ntl) { all = false; break; }
          }
          if (!all) break;
          for (int r = 0; r < C; ++r) {
            const Task& u = lists[base + r][pc[base + r]];
            for (int j = 0; j < u.ntl; ++j) cnt[tile_signal(p.s, u, j)]++;
            pc[base + r]++;
            remaining--;
          }
        } else {
          cnt[t.signal]++; pc[b]++; remaining--;
        }
        progress = true;
      }
    }
  }
  if (remaining) {
    for (int b = 0; b < G; ++b)
      if (pc[b] < lists[b].size()) {
        const Task& t = lists[b][pc[b]];
        fmt(msg, msglen, "deadlock: CTA " + std::to_string(b) + " stuck at phase " + std::to_string(t.phase) +
                             " (" + std::to_string(remaining) + " tasks left)");
        break;
      }
    return 1;
  }
  (void)nph;
  fmt(msg, msglen, "ok");
  return 0;
}

}  // namespace cp
