// cp_internal.h -- structures shared by the host scheduler, the launcher and
// the frame kernel. Plain C++ (no CUDA types) so the scheduler and its checks
// compile and run without a GPU.
#pragma once
#include <stdint.h>
#include <stddef.h>

namespace cp {

// ---------------------------------------------------------------- constants
constexpr int kMaxRows = 128;          // rows one frame can carry: handles of up to 64 rows run
                                       // M = 64 MMAs, larger ones M = 128 (row i in TMEM lane i)
constexpr int kRowsM64 = 64;           // the most rows of an M = 64 handle
constexpr int kThreads = 320;          // warp 0 producer, warp 1 MMA, warps 2..9 compute
constexpr int kComputeBase = 64;       // first compute thread
constexpr int kComputeThreads = 256;
constexpr int kNumA = 8;               // activation K-chunk slots (64 rows x 128 B each); an
                                       // M = 128 handle pairs adjacent slots (128 rows, 16 KB)
constexpr int kNumW = 4;               // weight pages in the ring (one qkv / gate-up tile part)
constexpr int kPageBytes = 24576;      // one weight page: one K-chunk of the widest tile (192 x 128 B)
constexpr int kAChunkBytes = 8192;     // 64 rows x 64 bf16
constexpr int kRecvPad = 4;            // floats of padding per received row: senders' lanes are rows,
                                       // and a row stride that is not a multiple of 128 B keeps their
                                       // 16-byte stores on different banks
constexpr int kRecvPadH = 8;           // the same 16 bytes for the fp16 exchange of the normed kinds
constexpr int kMaxTileN = 192;         // widest tile (gate/up); fp32 partials only for N = 32 tiles
constexpr int kRecvBytes = kRowsM64 * (kMaxTileN + kRecvPadH) * 2;  // one partial-sum receive slot of an
                                                                     // M = 64 handle; an M = 128 handle
                                                                     // uses both as one slot
static_assert(kRecvBytes >= kRowsM64 * (32 + kRecvPad) * 4, "receive slot holds the fp32 exchange");
static_assert(2 * kRecvBytes >= kMaxRows * (kMaxTileN + kRecvPadH) * 2, "joined slot holds 128 rows");
constexpr int kCounterStride = 64;     // counters per phase: one per 64-feature chunk of x (the
                                       // input projection, o, down), per gate/up tile, per kv
                                       // group (qkv, attention), or one (heads, draws, first
                                       // embedding)
constexpr int kMaxPositions = 16;
constexpr int kMaxVocab = 2048;
constexpr int kRowBlock = 8;           // rows per attention task
constexpr int kTraceStamps = 16;

// Shared-memory layout of the frame kernel (offsets from a 1024-aligned base).
constexpr int kSmemA = 0;
constexpr int kSmemW = kSmemA + kNumA * kAChunkBytes;            // the MMAs (M = 64) read
                                                                 // each A slot as one 64-row
                                                                 // tile: nothing past a slot
                                                                 // is read
constexpr int kSmemRecv = kSmemW + kNumW * kPageBytes;
constexpr int kSmemMisc = kSmemRecv + 2 * kRecvBytes;
constexpr int kSmemMiscBytes = 2048;
constexpr int kSmemBytes = kSmemMisc + kSmemMiscBytes + 1024;    // + alignment slack

// Task types.
enum TaskType : int32_t { T_PROJ = 1, T_ATTN = 2, T_DRAW = 3, T_EMB0 = 4 };
// Projection kinds (also the phase kinds); ATTN/DRAW/EMB0 reuse the numbering.
enum Kind : int32_t {
  K_INPROJ = 0, K_EMB0 = 1, K_QKV = 2, K_ATTN = 3, K_O = 4, K_GU = 5, K_DOWN = 6,
  K_HEAD = 7, K_DRAW = 8
};

// One unit of work of one CTA. Projections are split along K over the CTAs of
// a cluster; every CTA of the cluster holds one part (kslice = its rank).
struct Task {
  int32_t type : 8;    // TaskType
  int32_t kind : 8;    // Kind
  int32_t kslice : 8;  // K part = cluster rank (projection)
  int32_t ntl : 8;     // projection: tiles in this task (1 or 2; tile, tile+1 share the staged K part)
  int32_t layer;     // transformer layer (qkv/attn/o/gu/down)
  int32_t pos;       // depth position whose residual stream is read/written
  int32_t group;     // head index (head/draw), kv group (attn), -1 otherwise
  int32_t tile;      // output tile (projection), row block (attn), row (draw/emb0)
  int32_t nfeat;     // output features of the tile (MMA N)
  int32_t k0;        // first input element of this K part
  int32_t nkc;       // 64-element K chunks in this part
  int32_t cpp;       // K chunks per weight page
  int32_t phase;     // phase index in the frame
  int32_t wait0, target0, wait1, target1;   // counters to wait for (-1: none)
  int32_t signal;    // counter to bump when done (first tile)
  int32_t cbase;     // per-chunk waits: counter of the producer phase's slot 0 (-1: none). Input
                     // chunk c (64 elements of K) waits for slots (64c) / fps .. (64c + 63) / fps
  int32_t cpack;     // per-chunk waits: target of each slot | fps << 16
  int32_t signal_b;  // counter the second tile of a two-tile task bumps (-1: none)
  int64_t w_off;     // byte offset of this part's packed weights
};
static_assert(sizeof(Task) == 80 && sizeof(Task) % 16 == 0, "task record size");

// Phase descriptor (host).
struct Phase {
  int kind, layer, pos, group;
  int ntiles, nfeat, K;       // projections
  int64_t w_base;             // packed weight offset of the tile grid
};

// Model shape as the scheduler sees it.
struct Shape {
  int L, H, Hq, Hkv, D, F, P, V, T, MR;
  float eps, rope_base;
  int qk_norm;
};

// The Qwen3-TTS 1.7B CodePredictor's sizes ("Qwen3-TTS: Run the 1.7B Depth
// Loop as One Persistent Kernel on Hopper": 5 layers, hidden 1024, 16/8 heads
// of 128, FFN 3072, 16 positions, vocabulary 2048, input projection from the
// 2048-wide talker) and the 4-CTA cluster: the frame kernel's specialised
// build fixes them at compile time; the host runs it for a handle whose shape
// and cluster match, and the shape-generic build otherwise. (The rows a handle
// holds, eps and the RoPE base stay parameters.)
struct FixedShape {
  int L, H, Hq, Hkv, D, F, P, V, T, qk_norm, cluster;
};
constexpr FixedShape kShape1p7b = {5, 1024, 16, 8, 128, 3072, 16, 2048, 2048, 1, 4};

// Per-frame arguments (device-visible).
struct FrameArgs {
  const float* h;            // [rows][T]
  const int32_t* c0;         // [rows]
  const float* temperature;  // [rows]
  const int32_t* top_k;
  const float* top_p;
  const uint64_t* seed;
  int64_t* offset;
  int32_t* codes;            // [rows][P-1]
  float* emb_sum;            // [rows][H] (may point to scratch)
  int rows;
  int write_emb_sum;
};

// Kernel parameters.
struct KParams {
  const Task* tasks;
  const int32_t* task_start;   // [grid+1]
  const int32_t* phase_start;  // [grid][nph+1]
  const uint8_t* wpack;
  const uint16_t* embed;       // [P][V][H] bf16
  const uint16_t* attn_norm;   // [L][H]
  const uint16_t* mlp_norm;
  const uint16_t* q_norm;      // [L][D]
  const uint16_t* k_norm;
  const uint16_t* final_norm;  // [H]
  const float* rope;           // [P][D/2][2] cos, sin
  float* x;                    // [P][MR][H]
  float* ssq;                  // [P][MR][H/32]
  uint16_t* q;                 // [MR][Hq][D]
  uint16_t* kv;                // [L][Hkv][MR/8][P][8][2][D]: keys and values; one row block's
                               // positions 0..p are contiguous (one bulk copy per attention task)
  uint16_t* o;                 // [Hq*D/64][MR][64] swizzled chunks
  uint16_t* m;                 // [F/64][MR][64] swizzled chunks
  uint16_t* xb;                // [P][H/64][MR][64] swizzled chunks of bf16(x * gain of x's next norm)
  float* logits;               // [P-1][MR][V]
  uint32_t* counters;          // [nph][kCounterStride]
  int32_t* status;             // [0] status, [1] abort flag, [2] done count, [3..7] detail
  int64_t* trace;              // [tasks][8] or null
  const FrameArgs* fa_dev;     // split mode: frame arguments in device memory
  FrameArgs fa;                // persistent mode: frame arguments by value
  Shape s;
  float attn_scale;
  int cluster;
  int nph;
  int ncounters;
  int mode;                    // 0 persistent, 1 one phase (split graph)
  int m128;                    // M = 128 projections (a handle of more than 64 rows)
  int phase_lo, phase_hi;      // phases this launch runs
  int last_launch;             // reset counters at the end
  int64_t timeout_ns;
  int stall_task;              // global task index whose wait never ends (test), -1 off
  int stall_staging;           // test: the leader's first bulk staging waits for good (abort path)
};

// Host plan.
struct Plan;
int plan_build(const Shape& s, int grid, int cluster, bool chunk_waits, Plan** out, char* msg, int msglen);
int plan_check(const Plan* p, int corrupt, char* msg, int msglen);
void plan_free(Plan* p);

struct PlanView {
  const Task* tasks; int ntasks;
  const int32_t* task_start; int grid;
  const int32_t* phase_start; int nph;
  int ncounters;
  int64_t wpack_bytes;
  int64_t weight_bytes, max_cta_bytes, min_cta_bytes;
  int max_tasks_per_cta;
  const Phase* phases;
};
PlanView plan_view(const Plan* p);

// Where a projection's packed weight tile grid starts and how its tiles map
// onto the source matrix rows (used by the packer).
int proj_nfeat(const Shape& s, int kind);
int proj_k(const Shape& s, int kind);
int proj_ntiles(const Shape& s, int kind);

}  // namespace cp
