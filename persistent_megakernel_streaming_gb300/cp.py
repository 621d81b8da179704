"""ctypes binding of libcp.so (include/cp.h): argument marshalling only.

Every step of the frame runs in the library's CUDA kernels; this module only
turns torch tensors into raw pointers and stream handles and maps status codes
to exceptions. It fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libcp.so")

CP_OK = 0
STATUS = {0: "CP_OK", 1: "CP_ERR_INVALID_ARG", 2: "CP_ERR_UNSUPPORTED", 3: "CP_ERR_RESIDENCY",
          4: "CP_ERR_CUDA", 5: "CP_ERR_TIMEOUT", 6: "CP_ERR_DEVICE_BOUNDS", 7: "CP_ERR_NOMEM",
          8: "CP_ERR_PLAN", 9: "CP_ERR_SCRATCH_LIMIT", 10: "CP_ERR_RANGE"}
CP_ERR_TIMEOUT = 5
CP_ERR_PLAN = 8
CP_ERR_SCRATCH_LIMIT = 9
CP_ERR_RANGE = 10

EXPORTS = ["cp_create", "cp_frame", "cp_frame_split", "cp_debug_logits", "cp_debug_state", "cp_status",
           "cp_clear_status", "cp_get_info", "cp_trace", "cp_destroy", "cp_strerror",
           "cp_plan_check", "cp_test_philox", "cp_test_draw", "cp_frame_static"]


class Shape(C.Structure):
    _fields_ = [("layers", C.c_int), ("hidden", C.c_int), ("q_heads", C.c_int), ("kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn", C.c_int), ("positions", C.c_int), ("vocab", C.c_int),
                ("talker_hidden", C.c_int), ("max_rows", C.c_int), ("rms_eps", C.c_float),
                ("rope_base", C.c_float), ("qk_norm", C.c_int)]


_PP = C.POINTER(C.c_void_p)


class Weights(C.Structure):
    _fields_ = [("in_proj", C.c_void_p), ("embed", _PP), ("attn_norm", _PP), ("mlp_norm", _PP),
                ("q_norm", _PP), ("k_norm", _PP), ("w_qkv", _PP), ("w_o", _PP), ("w_gate", _PP),
                ("w_up", _PP), ("w_down", _PP), ("final_norm", C.c_void_p), ("heads", _PP)]


class Sampler(C.Structure):
    _fields_ = [("temperature", C.c_void_p), ("top_k", C.c_void_p), ("top_p", C.c_void_p),
                ("seed", C.c_void_p), ("offset", C.c_void_p)]


class Options(C.Structure):
    _fields_ = [("cluster", C.c_int), ("max_ctas", C.c_int), ("timeout_ns", C.c_int64), ("trace", C.c_int),
                ("n_cuts", C.c_int), ("cuts", C.POINTER(C.c_int)), ("debug_stall_task", C.c_int),
                ("debug_stall_staging", C.c_int), ("generic_kernel", C.c_int), ("phase_waits", C.c_int)]


class Info(C.Structure):
    _fields_ = [("grid", C.c_int), ("cluster", C.c_int), ("threads", C.c_int), ("smem_bytes", C.c_int),
                ("phases", C.c_int), ("tasks", C.c_int), ("weight_bytes", C.c_int64),
                ("max_cta_weight_bytes", C.c_int64), ("min_cta_weight_bytes", C.c_int64),
                ("scratch_bytes", C.c_int64), ("sm_count", C.c_int), ("specialized", C.c_int)]


class PlanStats(C.Structure):
    _fields_ = [("phases", C.c_int), ("tasks", C.c_int), ("counters", C.c_int), ("weight_bytes", C.c_int64),
                ("max_cta_weight_bytes", C.c_int64), ("min_cta_weight_bytes", C.c_int64),
                ("max_tasks_per_cta", C.c_int), ("message", C.c_char * 160)]


class CPError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "persistent_megakernel_streaming_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        vp, i, st = C.c_void_p, C.c_int, C.c_void_p
        L.cp_create.argtypes = [C.POINTER(Shape), C.POINTER(Weights), i, C.POINTER(Options), C.POINTER(vp)]
        for name in ("cp_frame", "cp_frame_split", "cp_frame_static"):
            getattr(L, name).argtypes = [vp, vp, vp, C.POINTER(Sampler), i, vp, vp, st]
        L.cp_debug_logits.argtypes = [vp, i, vp, st]
        L.cp_debug_state.argtypes = [vp, i, i, i, vp, st]
        L.cp_status.argtypes = [vp]
        L.cp_clear_status.argtypes = [vp]
        L.cp_get_info.argtypes = [vp, C.POINTER(Info)]
        L.cp_trace.argtypes = [vp, vp, st]
        L.cp_destroy.argtypes = [vp]
        L.cp_destroy.restype = None
        L.cp_strerror.argtypes = [i]
        L.cp_strerror.restype = C.c_char_p
        L.cp_plan_check.argtypes = [C.POINTER(Shape), i, i, i, i, C.POINTER(PlanStats)]
        L.cp_test_philox.argtypes = [vp, vp, i, i, vp, st]
        L.cp_test_draw.argtypes = [vp, i, i, C.POINTER(Sampler), i, vp, st]
        _lib = L
    return _lib


def _check(code: int, what: str):
    if code != CP_OK:
        raise CPError(code, what)


def make_shape(d: dict) -> Shape:
    return Shape(d["layers"], d["hidden"], d["q_heads"], d["kv_heads"], d["head_dim"], d["ffn"],
                 d["positions"], d["vocab"], d["talker_hidden"], d.get("max_rows", 64),
                 float(d["rms_eps"]), float(d["rope_base"]), int(d["qk_norm"]))


def plan_check(shape: dict, grid: int, cluster: int, corrupt: int = 0, chunk_waits: bool = False):
    """Host-only schedule build and check (no GPU). Returns (status, stats)."""
    ps = PlanStats()
    code = lib().cp_plan_check(C.byref(make_shape(shape)), grid, cluster, int(chunk_waits), corrupt, C.byref(ps))
    return code, ps


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


def _sampler(samp: dict) -> Sampler:
    return Sampler(_ptr(samp["temperature"]), _ptr(samp["top_k"]), _ptr(samp["top_p"]),
                   _ptr(samp["seed"]), _ptr(samp["offset"]))


class Frame:
    """A handle (cp_create) with the frame calls bound to torch tensors.

    ``weights``: dict of tensors (host or device) holding bf16 bit patterns in
    the layouts of include/cp.h (per-layer / per-position lists as stacked
    leading dimensions)."""

    def __init__(self, shape: dict, weights: dict, device: int = 0, cluster: int = 0, max_ctas: int = 0,
                 timeout_ns: int = 0, trace: bool = False, cuts=None, debug_stall_task: int = 0,
                 debug_stall_staging: bool = False, generic_kernel: bool = False, phase_waits: bool = False):
        self.shape = dict(shape)
        L, P = shape["layers"], shape["positions"]
        keep = []

        def one(t):
            keep.append(t)
            return C.c_void_p(_ptr(t))

        def many(t, n):
            arr = (C.c_void_p * n)(*[_ptr(t[i]) for i in range(n)])
            keep.append(t)
            keep.append(arr)
            return C.cast(arr, _PP)

        w = Weights(one(weights["in_proj"]), many(weights["embed"], P), many(weights["attn_norm"], L),
                    many(weights["mlp_norm"], L), many(weights["q_norm"], L), many(weights["k_norm"], L),
                    many(weights["w_qkv"], L), many(weights["w_o"], L), many(weights["w_gate"], L),
                    many(weights["w_up"], L), many(weights["w_down"], L), one(weights["final_norm"]),
                    many(weights["heads"], P - 1))
        cuts = list(cuts or [])
        cut_arr = (C.c_int * max(1, len(cuts)))(*cuts)
        opt = Options(cluster, max_ctas, timeout_ns, int(trace), len(cuts), cut_arr, debug_stall_task,
                      int(debug_stall_staging), int(generic_kernel), int(phase_waits))
        h = C.c_void_p()
        _check(lib().cp_create(C.byref(make_shape(shape)), C.byref(w), device, C.byref(opt), C.byref(h)),
               "cp_create")
        self._h = h
        self.info = Info()
        _check(lib().cp_get_info(h, C.byref(self.info)), "cp_get_info")

    def _call(self, fn, h, c0, samp, rows, codes, emb_sum, stream):
        sp = _sampler(samp)
        _check(fn(self._h, _ptr(h), _ptr(c0), C.byref(sp), int(rows), _ptr(codes), _ptr(emb_sum),
                  _stream(stream)), fn.__name__)

    def frame(self, h, c0, samp, rows, codes, emb_sum=None, stream=None):
        self._call(lib().cp_frame, h, c0, samp, rows, codes, emb_sum, stream)

    def frame_split(self, h, c0, samp, rows, codes, emb_sum=None, stream=None):
        self._call(lib().cp_frame_split, h, c0, samp, rows, codes, emb_sum, stream)

    def frame_static(self, h, c0, samp, rows, codes, emb_sum=None, stream=None):
        """cp_frame with its working set in the library's static scratch array."""
        self._call(lib().cp_frame_static, h, c0, samp, rows, codes, emb_sum, stream)

    def debug_logits(self, group, dst, stream=None):
        _check(lib().cp_debug_logits(self._h, int(group), _ptr(dst), _stream(stream)), "cp_debug_logits")

    def debug_state(self, what, a, b, dst, stream=None):
        _check(lib().cp_debug_state(self._h, int(what), int(a), int(b), _ptr(dst), _stream(stream)),
               "cp_debug_state")

    def trace(self, dst, stream=None):
        _check(lib().cp_trace(self._h, _ptr(dst), _stream(stream)), "cp_trace")

    def status(self) -> int:
        return lib().cp_status(self._h)

    def clear_status(self):
        _check(lib().cp_clear_status(self._h), "cp_clear_status")

    def close(self):
        if getattr(self, "_h", None):
            lib().cp_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def test_philox(ctr, key, use_curand: bool, out, stream=None):
    n = ctr.shape[0]
    _check(lib().cp_test_philox(_ptr(ctr), _ptr(key), n, int(use_curand), _ptr(out), _stream(stream)),
           "cp_test_philox")


def test_draw(logits, samp: dict, group: int, codes, stream=None):
    rows, vocab = logits.shape
    sp = _sampler(samp)
    _check(lib().cp_test_draw(_ptr(logits), rows, vocab, C.byref(sp), int(group), _ptr(codes),
                              _stream(stream)), "cp_test_draw")
