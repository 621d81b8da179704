/*
 * cp.h -- C ABI of the depth-decoder frame library (libcp.so).
 *
 * One call runs one frame of a codec-TTS depth decoder on one GPU: an input
 * projection of the talker hidden state, a GQA transformer (RMSNorm, QK-Norm,
 * RoPE, SwiGLU) stepped over the frame's depth positions, one code head and
 * one draw per later position, and one embedding step per code. The phases
 * and their count (432 at the 1.7B CodePredictor shape) follow "Qwen3-TTS:
 * Run the 1.7B Depth Loop as One Persistent Kernel on Hopper", section "How
 * it works"; the layer is the Qwen3 layer of "The gaps between kernels: PDL
 * and megakernels", section "How large are the gaps: an estimate".
 *
 * Conventions for every call:
 *  - Pointers to device memory are marked "device"; a pointer marked "host or
 *    device" may be either (the library copies through unified addressing).
 *  - Calls that take a cudaStream_t are asynchronous on that stream and
 *    return as soon as the work is queued; their inputs and outputs must stay
 *    valid until the stream reaches them. A null stream is the legacy stream.
 *  - Every call returns a cp_status code (0 = CP_OK); cp_strerror names it.
 *  - A handle serves one stream at a time and is not thread-safe.
 *  - Weights are bfloat16, row-major [out][in] (the nn.Linear layout), passed
 *    as raw 16-bit patterns (const void*).
 */
#ifndef CP_H
#define CP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cp_stream_t; /* same type as cudaStream_t */

/* ------------------------------------------------------------------ status */
enum cp_status {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = 1,   /* null pointer, rows out of range, bad option  */
  CP_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels are built for,
                               or not an sm_103 device: run another path     */
  CP_ERR_RESIDENCY = 3,     /* the GPU cannot keep every CTA of the frame
                               resident at once (e.g. an MPS share): the
                               CTAs wait on each other, so all must be
                               resident ("Qwen3-TTS: Run the 1.7B Depth
                               Loop as One Persistent Kernel on Hopper",
                               section "How it works", the MPS bullet)       */
  CP_ERR_CUDA = 4,          /* a CUDA runtime call failed                    */
  CP_ERR_TIMEOUT = 5,       /* sticky: a device-side wait gave up            */
  CP_ERR_DEVICE_BOUNDS = 6, /* sticky: a code or index outside its range
                               reached the device (the access was skipped)   */
  CP_ERR_NOMEM = 7,         /* device or host allocation failed              */
  CP_ERR_PLAN = 8,          /* the static schedule failed validation         */
  CP_ERR_SCRATCH_LIMIT = 9, /* cp_frame_static: the frame's working set does
                               not fit the library's static scratch array    */
  CP_ERR_RANGE = 10         /* sticky: a K-split partial sum of a normed
                               projection (qkv, gate/up, heads), which travels
                               between the cluster's CTAs as fp16 after the
                               norm's row factor, was outside the fp16 range;
                               the frame stopped                             */
};

/* ------------------------------------------------------------------ shapes */
/* Model shape. Limits the kernels are built for (CP_ERR_UNSUPPORTED outside):
 * head_dim 64 or 128; q_heads 1, 2 or 4 times kv_heads; kv_heads <= 16;
 * 2 <= positions <= 16; vocab a multiple of 256, at most 2048; hidden at
 * most 2048, a multiple of 64 * cluster and of 128; ffn a multiple of 64, at
 * most 6144 (96 * 64; 4096 when not a multiple of 96); every projection's
 * input width (hidden, q_heads * head_dim, ffn, talker_hidden) a multiple of
 * 64 * cluster; 1 <= max_rows <= 128. A handle of up to 64 rows runs its
 * projections as M = 64 tensor-core tiles; one of more, as M = 128 tiles (a
 * 128-row frame, "Qwen3-TTS: Run the 1.7B Depth Loop as One Persistent
 * Kernel on Hopper", sections "Decisions and experiments" and "What's left
 * in the frame, open": the pages' kernel stops at 64 rows). */
typedef struct cp_shape {
  int layers;         /* transformer layers (5)                             */
  int hidden;         /* hidden size H (1024)                               */
  int q_heads;        /* query heads Hq (16)                                */
  int kv_heads;       /* key/value heads Hkv (8); q head h reads kv head
                         h / (Hq / Hkv)                                     */
  int head_dim;       /* D (128)                                            */
  int ffn;            /* SwiGLU intermediate size F (3072)                  */
  int positions;      /* depth positions P per frame (16); P-1 codes drawn  */
  int vocab;          /* codebook size V (2048)                             */
  int talker_hidden;  /* width of the talker hidden state T (2048)          */
  int max_rows;       /* largest row count a frame will be called with
                         (64; at most 128)                                  */
  float rms_eps;      /* RMSNorm epsilon (1e-6)                             */
  float rope_base;    /* RoPE base (10000)                                  */
  int qk_norm;        /* nonzero: per-head RMSNorm on q and k before RoPE   */
} cp_shape;

/* Weights. Arrays of per-layer / per-position pointers are host arrays whose
 * elements point to host or device memory. All are read once by cp_create,
 * which copies and repacks them into memory the handle owns; the caller may
 * free them when cp_create returns. */
typedef struct cp_weights {
  const void* in_proj;                /* [hidden][talker_hidden]            */
  const void* const* embed;           /* positions x [vocab][hidden]; table
                                         k embeds code k                    */
  const void* const* attn_norm;       /* layers x [hidden]                  */
  const void* const* mlp_norm;        /* layers x [hidden]                  */
  const void* const* q_norm;          /* layers x [head_dim] (if qk_norm)   */
  const void* const* k_norm;          /* layers x [head_dim] (if qk_norm)   */
  const void* const* w_qkv;           /* layers x [(Hq+2Hkv)*D][hidden],
                                         rows q (head-major) | k | v        */
  const void* const* w_o;             /* layers x [hidden][Hq*D]            */
  const void* const* w_gate;          /* layers x [ffn][hidden]             */
  const void* const* w_up;            /* layers x [ffn][hidden]             */
  const void* const* w_down;          /* layers x [hidden][ffn]             */
  const void* final_norm;             /* [hidden]                           */
  const void* const* heads;           /* (positions-1) x [vocab][hidden];
                                         head j draws code j+1              */
} cp_weights;

/* Per-row sampler settings, all device arrays of length rows. A row draws
 * with temperature <= 0 as argmax (ties to the lowest index). Otherwise
 * logits are divided by the temperature; top_k in [1, vocab) keeps the k
 * best tokens (ties by lower index), 0 or >= vocab keeps all; top_p < 1
 * keeps tokens while the softmax mass of better kept tokens is below top_p
 * (the best is always kept); the code is the Gumbel-max over the kept set
 * with Philox4x32-10 uniforms keyed by (seed, row, offset + group).
 * offset is read and then advanced by positions-1 for every row.
 * ("Qwen3-TTS: Run the 1.7B Depth Loop ...", section "How it works": the
 * kernel reads each row's temperature, top-k, top-p, seed and offset, and
 * moves the offsets as that many sample calls would.) */
typedef struct cp_sampler {
  const float* temperature;   /* device [rows]                              */
  const int32_t* top_k;       /* device [rows]                              */
  const float* top_p;         /* device [rows]                              */
  const uint64_t* seed;       /* device [rows]                              */
  int64_t* offset;            /* device [rows], read and advanced in place  */
} cp_sampler;

/* Options; pass NULL for defaults. */
typedef struct cp_options {
  int cluster;            /* CTAs per cluster for the K-split projections:
                             2, 4 or 8 (0 = default 4)                       */
  int max_ctas;           /* cap on the persistent grid (0 = every cluster
                             that can be resident)                           */
  int64_t timeout_ns;     /* give up a device-side wait after this long
                             (0 = default 2 s); the frame then ends with the
                             sticky CP_ERR_TIMEOUT                           */
  int trace;              /* nonzero: record per-task timestamps (cp_trace) */
  int n_cuts;             /* cp_frame only: split the persistent launch into
                             n_cuts+1 consecutive launches ...               */
  const int* cuts;        /* ... before these phase indices (ascending,
                             in (0, phases)); host array                     */
  int debug_stall_task;   /* testing: -1 or 0 = off; k > 0 makes the k-th
                             task of CTA 0 wait for a count nothing reaches,
                             so the frame ends with CP_ERR_TIMEOUT           */
  int debug_stall_staging; /* testing: nonzero makes every CTA's leader wait
                             for a count nothing reaches when it stages its
                             first bulk-copied K part (the abort path of the
                             staging, one thread per CTA), so the frame ends
                             with CP_ERR_TIMEOUT                             */
  int generic_kernel;     /* testing: nonzero runs the shape-generic build of
                             the frame kernel even where the shape has a
                             specialised one (cp_info.specialized)           */
  int phase_waits;        /* nonzero: every projection waits for its whole
                             producer phase (one counter) before it stages
                             any input. By default it waits per K chunk
                             ("Qwen3-TTS: Run the 1.7B Depth Loop as One
                             Persistent Kernel on Hopper", section "What's
                             left in the frame, open"): each 64-element input
                             chunk is staged as soon as the producer tiles of
                             that chunk are done (the producers signal one
                             counter per chunk, per gate/up tile or per kv
                             group). Same results bit for bit; per-chunk
                             waits measured 1.4 % faster at 64 and 128 rows */
} cp_options;

typedef struct cp_handle cp_handle; /* opaque, owned by the library */

/* Build a handle on `device`: validate the shape and the device (sm_103,
 * every CTA resident), copy and repack the weights into handle-owned device
 * memory (projection weights as pre-swizzled K-chunks in the order the
 * schedule streams them), allocate the frame's scratch, build and validate
 * the static per-CTA task schedule. The current device is restored on
 * return. *out is set only on CP_OK. Errors: CP_ERR_INVALID_ARG (null or
 * unreadable pointer, bad option), CP_ERR_UNSUPPORTED (shape or device),
 * CP_ERR_RESIDENCY, CP_ERR_NOMEM, CP_ERR_PLAN, CP_ERR_CUDA; nothing is
 * leaked on failure.
 * ("Qwen3-TTS: Run the 1.7B Depth Loop as One Persistent Kernel on Hopper":
 * section "How it works" for the static per-CTA task list built on the host
 * and the residency rule; the review discussion for the set-up's parts,
 * weight stacking and scratch allocation, done once per handle.) */
int cp_create(const cp_shape* shape, const cp_weights* weights, int device,
              const cp_options* options, cp_handle** out);

/* One frame as one persistent launch (or n_cuts+1 launches when cut):
 * "Qwen3-TTS: Run the 1.7B Depth Loop as One Persistent Kernel on Hopper",
 * section "How it works" (one launch walks the frame's 432 phases; the
 * kernel draws in place and moves the offsets as that many sample calls
 * would). Inputs and outputs are caller-owned device memory.
 *  talker_hidden  device fp32 [rows][talker_hidden]
 *  first_code     device int32 [rows], each in [0, vocab)
 *  sampler        per-row settings (device arrays); offset advanced
 *  rows           1 <= rows <= max_rows
 *  codes_out      device int32 [rows][positions-1]: codes 1..P-1
 *  emb_sum_out    device fp32 [rows][hidden] or NULL: sum over the frame's
 *                 P codes of their embeddings, added in code order
 * Results are bit-identical run to run and to cp_frame_split; a row's
 * results do not depend on the other rows. Errors: CP_ERR_INVALID_ARG (null
 * pointer, rows outside [1, max_rows]), CP_ERR_CUDA (the launch failed);
 * device-side errors are sticky and read with cp_status. */
int cp_frame(cp_handle* h, const float* talker_hidden, const int32_t* first_code,
             const cp_sampler* sampler, int rows, int32_t* codes_out,
             float* emb_sum_out, cp_stream_t stream);

/* The same frame with the same tiles, as one kernel per phase, replayed from
 * a CUDA Graph with programmatic dependent launch between the kernels (each
 * kernel streams its weights before it waits for the previous one). The
 * graph is built on the first call. Same arguments and results as cp_frame.
 * ("The gaps between kernels: PDL and megakernels", section "PDL: letting
 * the next kernel start early".) */
int cp_frame_split(cp_handle* h, const float* talker_hidden, const int32_t* first_code,
                   const cp_sampler* sampler, int rows, int32_t* codes_out,
                   float* emb_sum_out, cp_stream_t stream);

/* Bytes of device memory the library reserves, once per device that loads
 * it, as a static array for cp_frame_static; held until the process exits. */
#define CP_STATIC_SCRATCH_BYTES (16u << 20)

/* cp_frame without any device allocation behind it. The paper has no
 * counterpart to this call.
 *
 * Some callers cannot allocate device memory where they run a frame: code
 * working inside an open stream capture (cudaMalloc is refused there), under
 * an allocator that owns all device memory, or on a thread that must not
 * block while cudaMalloc waits for the device. cp_frame itself allocates
 * nothing, but its per-frame working set (residual stream, frame K/V cache,
 * activations, logits, dependency counters) was allocated by cp_create for
 * the handle; this call instead takes that working set from a static array
 * of CP_STATIC_SCRATCH_BYTES that the library reserves on every device that
 * loads it. The handle supplies its packed weights, its schedule and its
 * status words; arguments, results and bit-identity with cp_frame are as for
 * cp_frame.
 *
 * Limit: the working set grows with rows, with the frame K/V cache carved in
 * blocks of 8 rows; at the 1.7B CodePredictor shape (5 layers, hidden 1024,
 * 16/8 heads of 128, FFN 3072, 16 positions, vocabulary 2048) 25 rows fit
 * (16.64 MB) and 26 do not (16.88 MB). A call whose rows do not fit returns
 * CP_ERR_SCRATCH_LIMIT without launching anything.
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, once per device) with that device current; make
 * that first call before any stream capture starts.
 * Sharing: every call uses the one array, which keeps the last call's
 * contents; each call clears its dependency counters before it launches.
 * Calls that overlap on the GPU (two streams, or two handles) race and must
 * not be issued.
 * Errors: device-side errors go to the handle's sticky status, as for
 * cp_frame (cp_status reads it; while it is set, this call and cp_frame
 * return at once without computing). The handle's test stalls
 * (debug_stall_task, debug_stall_staging) apply here too.
 * cp_debug_logits and cp_debug_state read the handle's working set, so they
 * show the last cp_frame or cp_frame_split of the handle, not this call. */
int cp_frame_static(cp_handle* h, const float* talker_hidden, const int32_t* first_code,
                    const cp_sampler* sampler, int rows, int32_t* codes_out,
                    float* emb_sum_out, cp_stream_t stream);

/* Copy the logits of head `group` (0 <= group < positions-1) from the last
 * frame run on this handle: device fp32 [rows][vocab] of that frame
 * (caller-owned, asynchronous on `stream`; CP_ERR_INVALID_ARG for a bad
 * group or before any frame). It serves the check "the frame against the
 * loop with given codes: ... logits stay within ... of the largest logit"
 * ("Qwen3-TTS: Run the 1.7B Depth Loop ...", section "Testing"). */
int cp_debug_logits(cp_handle* h, int group, float* dst, cp_stream_t stream);

/* Copy part of the last frame's internal state, for phase-by-phase checks:
 *  what 0: position a's residual stream at the end of the frame (its output
 *          after every layer), device fp32 [rows][hidden];
 *  what 1: the keys layer a wrote at position b (after QK-Norm and RoPE),
 *          device bf16 [rows][kv_heads][head_dim];
 *  what 2: the values layer a wrote at position b, same layout. */
int cp_debug_state(cp_handle* h, int what, int a, int b, void* dst, cp_stream_t stream);

/* Synchronise the device and return the handle's sticky device status
 * (CP_OK, CP_ERR_TIMEOUT, CP_ERR_DEVICE_BOUNDS or CP_ERR_RANGE; CP_ERR_CUDA
 * if the synchronisation itself fails). While it is not CP_OK, frames
 * return at once without computing. The waits it reports are the bounded
 * form of the dependency waits of "The gaps between kernels: PDL and
 * megakernels", section "Megakernels" (a task that waits for an earlier one
 * can only deadlock if that one never runs: here it gives up instead). */
int cp_status(cp_handle* h);

/* Synchronise the device and reset the sticky status and the frame state. */
int cp_clear_status(cp_handle* h);

/* Launch geometry and plan statistics of a handle. */
typedef struct cp_info {
  int grid;            /* CTAs of the persistent launch                     */
  int cluster;         /* CTAs per cluster                                  */
  int threads;         /* threads per CTA                                   */
  int smem_bytes;      /* dynamic shared memory per CTA                     */
  int phases;          /* phases per frame                                  */
  int tasks;           /* tasks per frame over all CTAs                     */
  int64_t weight_bytes;        /* projection weight bytes streamed per frame */
  int64_t max_cta_weight_bytes;/* the most any one CTA streams per frame    */
  int64_t min_cta_weight_bytes;/* the least                                 */
  int64_t scratch_bytes;       /* device scratch owned by the handle        */
  int sm_count;        /* SMs on the device                                 */
  int specialized;     /* 1: the frame kernel build with this shape's sizes
                          fixed at compile time runs (the Qwen3-TTS 1.7B
                          CodePredictor: L 5, hidden 1024, 16/8 heads of
                          128, FFN 3072, 16 positions, vocabulary 2048,
                          input 2048, clusters of 4); 0: the build that
                          reads every size at run time                     */
} cp_info;

int cp_get_info(const cp_handle* h, cp_info* out);

/* Per-task timestamps of the last frame run with options.trace set: device
 * int64 [info.tasks][16] of %globaltimer ns, in the order tasks appear in the
 * schedule (CTA-major). Compute warps: 0 task start, 1 dependencies
 * satisfied (with per-chunk waits: the first input chunk's producers seen
 * done), 2 inputs staged, 3 accumulator ready, 4 partial sums exchanged,
 * 5 outputs stored, 6 signal issued; word 7 packs (phase << 32) |
 * (kind << 16) | CTA. MMA warp: 8 accumulator free, 9 weights landed (last
 * page), 10 inputs ready (last chunk), 12 MMAs committed. Producer warp: 11
 * last weight page issued. Stamps a task type lacks are 0. */
int cp_trace(cp_handle* h, int64_t* dst, cp_stream_t stream);

/* Release everything the handle owns (synchronises its device): the
 * stacked weights, the scratch, the schedule and the split graph that
 * cp_create and the first cp_frame_split made ("Qwen3-TTS: Run the 1.7B
 * Depth Loop ...", review discussion: weight stacking and scratch
 * allocation). A null handle is ignored. */
void cp_destroy(cp_handle* h);

/* A static, human-readable name for a cp_status code ("unknown status" for
 * others). The codes are this library's; the conditions they name are the
 * refusals of "Qwen3-TTS: Run the 1.7B Depth Loop ...", section "How it
 * works" (a step the kernel cannot take runs the loop instead). */
const char* cp_strerror(int status);

/* ------------------------------------------------------------ host checks */
/* Build the static schedule for `shape` with `grid` CTAs in clusters of
 * `cluster`, without a GPU, and check it: every wait is matched by exactly
 * the signals of its phase, dependencies only point to earlier phases, the
 * parts of every K-split tile sit on one cluster with distinct ranks, and a
 * simulation of the per-CTA lists (cluster tasks meeting in lockstep) runs to
 * the end without deadlock. `chunk_waits` nonzero builds the schedule with
 * per-chunk waits (the handles' default), zero with whole-phase waits
 * (cp_options.phase_waits). `corrupt` is for testing the checker: 0 = none,
 * 1 = raise one wait target past its signals, 2 = move one task ahead of the
 * task it depends on in its CTA's list, 3 = give two parts of one tile the
 * same cluster rank. Returns CP_OK or CP_ERR_PLAN; fills *out if non-NULL. */
typedef struct cp_plan_stats {
  int phases;
  int tasks;
  int counters;
  int64_t weight_bytes;
  int64_t max_cta_weight_bytes;
  int64_t min_cta_weight_bytes;
  int max_tasks_per_cta;
  char message[160];   /* why a check failed */
} cp_plan_stats;

int cp_plan_check(const cp_shape* shape, int grid, int cluster, int chunk_waits, int corrupt,
                  cp_plan_stats* out);

/* ------------------------------------------------------------ test hooks */
/* Run the frame kernels' Philox4x32-10 on n (counter, key) pairs, or
 * cuRAND's curand_Philox4x32_10 when use_curand is nonzero. Device arrays:
 * ctr uint32 [n][4], key uint32 [n][2], out uint32 [n][4]. */
int cp_test_philox(const uint32_t* ctr, const uint32_t* key, int n, int use_curand,
                   uint32_t* out, cp_stream_t stream);

/* Run the frame kernels' draw on given logits: device fp32 [rows][vocab],
 * sampler arrays as in cp_sampler (offset only read: row r draws at
 * offset[r] + group), Philox row index = the row's index here. Writes device
 * int32 codes [rows]. 1 <= rows, vocab a multiple of 256 up to 2048. */
int cp_test_draw(const float* logits, int rows, int vocab, const cp_sampler* sampler,
                 int group, int32_t* codes, cp_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* CP_H */
