"""GB300 (sm_103a) FP4 block-scaled quantized linear layer.

Python face of libfp4bs.so (include/fp4bs.h). The functions below have the
C-ABI names and only marshal arguments: PyTorch tensors supply device memory,
PyTorch streams the CUDA stream, and every step of the quantizer and the GEMMs
runs in the library's kernels. Nothing here falls back to another
implementation: if the library is missing, calls raise.

Method: "Pretraining Large Language Models with NVFP4" (arXiv 2509.25149),
sections 4.1-4.4 and App. B-C, and the UE5M3 block-scale paper (arXiv
2609.02846). See include/fp4bs.h for the operation each entry point performs.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field

import torch

from . import _lib
from ._lib import (FP4_BLOCK_1x16, FP4_BLOCK_1x32, FP4_BLOCK_16x16, FP4_LAYOUT_PLAIN, FP4_LAYOUT_TCGEN05,
                   FP4_ORIENT_COLWISE, FP4_ORIENT_ROWWISE, FP4_ROUND_RNE, FP4_ROUND_SR, FP4_SCALE_E4M3,
                   FP4_SCALE_UE5M3, FP4_SCALE_UE8M0, FP4_TSCALE_CURRENT, FP4_TSCALE_GIVEN, FP4_TSCALE_HELD,
                   FP4_TSCALE_ROW,
                   Fp4Error)

__all__ = ["QTensor", "QuantConfig", "AmaxState", "fp4_quantize", "fp4_quantize_dual", "fp4_dequantize", "fp4_gemm",
           "fp4_gemm_workspace_bytes", "fp4_tensor_amax", "fp4_tensor_amax_dual", "fp4_linear_fprop", "fp4_linear_dgrad", "fp4_linear_wgrad", "fp4_device_status",
           "fp4_device_status_record", "fp4_workspace_bytes", "fp4_quantized_sizes", "row_stride", "Fp4Error",
           "Fp4Linear"]


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclass
class QTensor:
    """A quantized operand: rows x cols E2M1 codes (cols = dot dimension),
    block scales, and the FP32 decode tensor scale (one per row with per_row,
    the output of tscale FP4_TSCALE_ROW)."""
    codes: torch.Tensor
    scales: torch.Tensor
    s_dec: torch.Tensor
    rows: int
    cols: int
    scale_fmt: int = FP4_SCALE_E4M3
    block_k: int = 16
    layout: int = FP4_LAYOUT_TCGEN05
    per_row: bool = False

    @staticmethod
    def empty(rows: int, cols: int, scale_fmt: int = FP4_SCALE_E4M3, layout: int = FP4_LAYOUT_TCGEN05,
              device="cuda", per_row: bool = False) -> "QTensor":
        bk = 32 if scale_fmt == FP4_SCALE_UE8M0 else 16
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
        scales = torch.empty((rows * (cols // bk),), dtype=torch.uint8, device=device)
        # 16-byte multiples keep later buffers aligned
        n_sdec = (rows + 3) // 4 * 4 if per_row else 4
        s_dec = torch.empty((max(n_sdec, 4),), dtype=torch.float32, device=device)
        return QTensor(codes, scales, s_dec, rows, cols, scale_fmt, bk, layout, per_row)

    def desc(self) -> _lib.fp4_tensor_t:
        return _lib.fp4_tensor_t(self.codes.data_ptr(), self.scales.data_ptr(), self.s_dec.data_ptr(),
                                 self.rows, self.cols, self.scale_fmt, self.block_k, self.layout,
                                 int(self.per_row))


@dataclass
class QuantConfig:
    """Quantizer options (fp4_quant_params_t)."""
    scale_fmt: int = FP4_SCALE_E4M3
    block: int = FP4_BLOCK_1x16
    round: int = FP4_ROUND_RNE
    orient: int = FP4_ORIENT_ROWWISE
    rht: bool = False
    tscale: int = FP4_TSCALE_CURRENT
    target_T: float = 448.0
    refresh_every: int = 50
    tensor_id: int = 0
    layout: int = FP4_LAYOUT_TCGEN05
    emit_transpose: bool = False
    seed: int = 0
    step: int = 0

    def params(self) -> _lib.fp4_quant_params_t:
        return _lib.fp4_quant_params_t(self.scale_fmt, self.block, self.round, self.orient, int(self.rht),
                                       self.tscale, self.target_T, self.refresh_every, self.tensor_id,
                                       self.layout, int(self.emit_transpose), 0, self.seed, self.step)


class AmaxState:
    """Device-resident held-amax record (fp4_amax_state_t, 16 bytes)."""

    def __init__(self, device="cuda"):
        self.buf = torch.zeros(4, dtype=torch.int32, device=device)

    @property
    def amax(self) -> float:
        return float(self.buf[0:1].view(torch.float32).item())

    @property
    def valid(self) -> int:
        return int(self.buf[1].item())

    @property
    def last_refresh_step(self) -> int:
        return int(self.buf[2:4].view(torch.int64).item())


def fp4_quantized_sizes(cfg: QuantConfig, rows: int, cols: int) -> tuple[int, int]:
    c, s = ctypes.c_size_t(), ctypes.c_size_t()
    p = cfg.params()
    _lib.check(_lib.load().fp4_quantized_sizes(ctypes.byref(p), rows, cols, ctypes.byref(c), ctypes.byref(s)),
               "fp4_quantized_sizes")
    return c.value, s.value


def fp4_workspace_bytes(cfg: QuantConfig, rows: int, cols: int) -> int:
    p = cfg.params()
    return _lib.load().fp4_workspace_bytes(ctypes.byref(p), rows, cols)


def row_stride(x: torch.Tensor) -> int:
    """The row stride (ld, in elements) of a 2-D BF16 matrix whose rows are
    contiguous, e.g. a column slice of a wider buffer."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and (x.stride(1) == 1 or x.shape[1] <= 1), \
        "rows must be contiguous"
    return x.stride(0) if x.shape[0] > 1 else x.shape[1]


def fp4_quantize(cfg: QuantConfig, x: torch.Tensor, out: QTensor, out_t: QTensor | None = None,
                 state: AmaxState | None = None, counters: torch.Tensor | None = None,
                 ws: torch.Tensor | None = None, stream=None) -> None:
    """Quantize the row-major BF16 matrix `x` into `out` (see fp4_quantize in
    fp4bs.h); `x` may be a view whose rows lie further apart than its width."""
    ld = row_stride(x)
    p = cfg.params()
    d = out.desc()
    dt = out_t.desc() if out_t is not None else None
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    st = _lib.load().fp4_quantize(ctypes.byref(p), _ptr(x), x.shape[0], x.shape[1], ld, ctypes.byref(d),
                                  ctypes.byref(dt) if dt is not None else None,
                                  _ptr(state.buf) if state is not None else None, _ptr(counters), _ptr(ws),
                                  ws_bytes, _stream(stream))
    _lib.check(st, "fp4_quantize")


def fp4_quantize_dual(cfg_row: QuantConfig, cfg_col: QuantConfig, x: torch.Tensor, out_row: QTensor,
                      out_col: QTensor, state_row: AmaxState | None = None, state_col: AmaxState | None = None,
                      counters_row: torch.Tensor | None = None, counters_col: torch.Tensor | None = None,
                      ws: torch.Tensor | None = None, stream=None) -> None:
    """Rowwise and colwise quantization of `x` in one pass (see fp4_quantize_dual in fp4bs.h)."""
    ld = row_stride(x)
    pr, pc = cfg_row.params(), cfg_col.params()
    dr, dc = out_row.desc(), out_col.desc()
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    st = _lib.load().fp4_quantize_dual(ctypes.byref(pr), ctypes.byref(pc), _ptr(x), x.shape[0], x.shape[1], ld,
                                       ctypes.byref(dr), ctypes.byref(dc),
                                       _ptr(state_row.buf) if state_row is not None else None,
                                       _ptr(state_col.buf) if state_col is not None else None,
                                       _ptr(counters_row), _ptr(counters_col), _ptr(ws), ws_bytes, _stream(stream))
    _lib.check(st, "fp4_quantize_dual")


AMAX_WS_BYTES = 2 * 2048 * 4  # workspace of fp4_tensor_amax / fp4_tensor_amax_dual


def fp4_tensor_amax(cfg: QuantConfig, x: torch.Tensor, out: AmaxState, ws: torch.Tensor, stream=None) -> None:
    """Tensor amax of the operand `cfg` describes into `out` (fp4_tensor_amax in fp4bs.h), for a later
    fp4_quantize with tscale FP4_TSCALE_GIVEN."""
    ld = row_stride(x)
    p = cfg.params()
    _lib.check(_lib.load().fp4_tensor_amax(ctypes.byref(p), _ptr(x), x.shape[0], x.shape[1], ld, _ptr(out.buf),
                                           _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
               "fp4_tensor_amax")


def fp4_tensor_amax_dual(cfg_row: QuantConfig, cfg_col: QuantConfig, x: torch.Tensor, out_row: AmaxState,
                         out_col: AmaxState, ws: torch.Tensor, stream=None) -> None:
    """Rowwise and colwise operand amaxes of `x` from one read (fp4_tensor_amax_dual in fp4bs.h)."""
    ld = row_stride(x)
    pr, pc = cfg_row.params(), cfg_col.params()
    _lib.check(_lib.load().fp4_tensor_amax_dual(ctypes.byref(pr), ctypes.byref(pc), _ptr(x), x.shape[0], x.shape[1], ld,
                                                _ptr(out_row.buf), _ptr(out_col.buf), _ptr(ws),
                                                ws.numel() * ws.element_size(), _stream(stream)),
               "fp4_tensor_amax_dual")


def fp4_dequantize(t: QTensor, out: torch.Tensor, stream=None) -> None:
    assert out.is_contiguous() and out.dtype in (torch.float32, torch.bfloat16)
    d = t.desc()
    _lib.check(_lib.load().fp4_dequantize(ctypes.byref(d), _ptr(out), int(out.dtype == torch.float32),
                                          _stream(stream)), "fp4_dequantize")


def fp4_gemm_workspace_bytes(a: QTensor, b: QTensor) -> int:
    da, db = a.desc(), b.desc()
    return _lib.load().fp4_gemm_workspace_bytes(ctypes.byref(da), ctypes.byref(db))


def fp4_gemm(a: QTensor, b: QTensor, d: torch.Tensor, accumulate: bool = False, stream=None,
             ws: torch.Tensor | None = None) -> None:
    """D = A B^T (fp4_gemm); with ``ws`` (fp4_gemm_workspace_bytes(a, b) bytes of
    device memory) UE5M3 operands take the rebiased native path (fp4_gemm_ws)."""
    assert d.is_contiguous() and d.dtype in (torch.float32, torch.bfloat16)
    da, db = a.desc(), b.desc()
    L = _lib.load()
    if ws is None:
        _lib.check(L.fp4_gemm(ctypes.byref(da), ctypes.byref(db), _ptr(d), int(d.dtype == torch.float32),
                              int(accumulate), _stream(stream)), "fp4_gemm")
    else:
        _lib.check(L.fp4_gemm_ws(ctypes.byref(da), ctypes.byref(db), _ptr(d), int(d.dtype == torch.float32),
                                 int(accumulate), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
                   "fp4_gemm_ws")


def fp4_linear_fprop(x: QTensor, w: QTensor, y: torch.Tensor, stream=None) -> None:
    dx, dw = x.desc(), w.desc()
    _lib.check(_lib.load().fp4_linear_fprop(ctypes.byref(dx), ctypes.byref(dw), _ptr(y), _stream(stream)),
               "fp4_linear_fprop")


def fp4_linear_dgrad(dy: QTensor, wt: QTensor, dx: torch.Tensor, stream=None) -> None:
    a, b = dy.desc(), wt.desc()
    _lib.check(_lib.load().fp4_linear_dgrad(ctypes.byref(a), ctypes.byref(b), _ptr(dx), _stream(stream)),
               "fp4_linear_dgrad")


def fp4_linear_wgrad(dyt: QTensor, xt: QTensor, dw: torch.Tensor, accumulate: bool = False, stream=None) -> None:
    a, b = dyt.desc(), xt.desc()
    _lib.check(_lib.load().fp4_linear_wgrad(ctypes.byref(a), ctypes.byref(b), _ptr(dw), int(accumulate),
                                            _stream(stream)), "fp4_linear_wgrad")


def fp4_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the bounded-wait self-test (fp4_selftest_wait_timeout in fp4bs.h)."""
    _lib.check(_lib.load().fp4_selftest_wait_timeout(limit_us, _stream(stream)), "fp4_selftest_wait_timeout")


def fp4_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word."""
    return _lib.load().fp4_device_status(_stream(stream))


def fp4_device_status_record(dst: torch.Tensor, stream=None) -> None:
    """In stream order, write the device status word into dst[0] (int32, device
    or pinned host memory) and clear it, without synchronising
    (fp4_device_status_record in fp4bs.h)."""
    assert dst.dtype == torch.int32 and dst.numel() >= 1
    _lib.check(_lib.load().fp4_device_status_record(_ptr(dst), _stream(stream)), "fp4_device_status_record")


# --------------------------------------------------------------------------- linear layer
def _mark(mark, label: str) -> None:
    if mark is not None:
        mark(label)


@dataclass
class Fp4Linear:
    """One FP4 quantized linear layer Y = X W^T with its backward GEMMs
    ("Pretraining LLMs with NVFP4", section 4.1, Fig. 5 and the recipe of
    section 4: 16x16 weight scales, 1x16 activation/gradient scales, SR on
    gradients, RHT16 on the Wgrad inputs). Owns the quantized buffers; each call
    of `step` runs five quantizations and three GEMMs through the C ABI.

    scale_fmt E4M3 gives NVFP4 with current tensor scaling; UE5M3 gives the
    UE5M3 recipe (held amax refreshed every `refresh_every` steps with target T,
    no RHT), whose GEMMs take the rebiased native path (fp4_gemm_ws) when
    `ue5m3_native` is set, else the emulated one.

    With current scaling and `overlap_amax` set (and T, K, N multiples of 128),
    the tensor amaxes of W, X and dY are computed on a second stream
    (fp4_tensor_amax) while the caller's stream quantizes W, X and dY in turn,
    each with its amax (FP4_TSCALE_GIVEN) as soon as that is ready: the same
    bytes as current scaling, with the amax passes off the critical path except
    W's (the smallest)."""
    tokens: int
    k_in: int
    n_out: int
    scale_fmt: int = FP4_SCALE_E4M3
    rht: bool = True
    seed: int = 0
    layer: int = 0
    target_T: float = 448.0
    held: bool = False
    refresh_every: int = 50
    ue5m3_native: bool = True
    overlap_amax: bool = True
    device: str = "cuda"
    bufs: dict = field(default_factory=dict)

    def __post_init__(self):
        T, K, N, f, dev = self.tokens, self.k_in, self.n_out, self.scale_fmt, self.device
        self.bufs = {
            "x": QTensor.empty(T, K, f, device=dev),        # X rowwise      (Fprop A)
            "w": QTensor.empty(N, K, f, device=dev),        # W 16x16        (Fprop B)
            "wt": QTensor.empty(K, N, f, device=dev),       # W^T 16x16      (Dgrad B)
            "dy": QTensor.empty(T, N, f, device=dev),       # dY rowwise SR  (Dgrad A)
            "dyt": QTensor.empty(N, T, f, device=dev),      # dY^T colwise   (Wgrad A)
            "xt": QTensor.empty(K, T, f, device=dev),       # X^T colwise    (Wgrad B)
        }
        self.ws = torch.empty(2 * fp4_workspace_bytes(QuantConfig(), 1, 1) // 4 + 4, dtype=torch.float32,
                              device=dev)
        self.counters = torch.zeros((5, 4), dtype=torch.int64, device=dev)
        self.states = [AmaxState(dev) for _ in range(5)] if self.held else [None] * 5
        self.side = None
        if self.overlap_amax and not self.held and T % 128 == 0 and K % 128 == 0 and N % 128 == 0:
            self.side = torch.cuda.Stream(device=dev)
            # one workspace per amax call: calls in flight must not share one
            self.ws_side = [torch.empty(AMAX_WS_BYTES // 4, dtype=torch.float32, device=dev) for _ in range(3)]
            self.given = [AmaxState(dev) for _ in range(5)]
            self.ev_inputs = torch.cuda.Event()
            self.ev_amax = [torch.cuda.Event() for _ in range(3)]
        self.gemm_ws = None
        if f == FP4_SCALE_UE5M3 and self.ue5m3_native:
            b = self.bufs
            need = max(fp4_gemm_workspace_bytes(b["x"], b["w"]), fp4_gemm_workspace_bytes(b["dy"], b["wt"]),
                       fp4_gemm_workspace_bytes(b["dyt"], b["xt"]))
            self.gemm_ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def _cfg(self, idx: int, step: int, **kw) -> QuantConfig:
        base = dict(scale_fmt=self.scale_fmt, target_T=self.target_T, seed=self.seed,
                    tensor_id=8 * self.layer + idx, step=step, refresh_every=self.refresh_every,
                    tscale=FP4_TSCALE_HELD if self.held else FP4_TSCALE_CURRENT)
        base.update(kw)
        return QuantConfig(**base)

    def quantize_all(self, x: torch.Tensor, w: torch.Tensor, dy: torch.Tensor, step: int = 0, stream=None,
                     mark=None):
        """X -> X (rowwise) and X^T (colwise + RHT) in one pass; W -> W and W^T
        (16x16); dY -> dY (rowwise, SR) and dY^T (colwise + RHT, SR) in one pass.
        Falls back to separate calls for shapes the one-pass kernel does not take.
        `mark`, if given, is called with a label before ("x") and after
        ("x/end") each call issued on the caller's stream (for timing)."""
        b, c = self.bufs, self.counters
        rht = self.rht
        dual_ok = self.tokens % 128 == 0 and self.k_in % 128 == 0 and self.n_out % 128 == 0
        if self.side is not None:
            self._quantize_all_overlapped(x, w, dy, step, stream, mark)
            return
        _mark(mark, "x")
        if dual_ok:
            fp4_quantize_dual(self._cfg(0, step), self._cfg(1, step, orient=FP4_ORIENT_COLWISE, rht=rht), x,
                              b["x"], b["xt"], self.states[0], self.states[1], c[0], c[1], ws=self.ws,
                              stream=stream)
        else:
            fp4_quantize(self._cfg(0, step), x, b["x"], state=self.states[0], counters=c[0], ws=self.ws,
                         stream=stream)
            fp4_quantize(self._cfg(1, step, orient=FP4_ORIENT_COLWISE, rht=rht), x, b["xt"], state=self.states[1],
                         counters=c[1], ws=self.ws, stream=stream)
        _mark(mark, "x/end")
        _mark(mark, "w")
        fp4_quantize(self._cfg(2, step, block=FP4_BLOCK_16x16, emit_transpose=True), w, b["w"], b["wt"],
                     state=self.states[2], counters=c[2], ws=self.ws, stream=stream)
        _mark(mark, "w/end")
        _mark(mark, "dy")
        if dual_ok:
            fp4_quantize_dual(self._cfg(3, step, round=FP4_ROUND_SR),
                              self._cfg(4, step, orient=FP4_ORIENT_COLWISE, rht=rht, round=FP4_ROUND_SR), dy,
                              b["dy"], b["dyt"], self.states[3], self.states[4], c[3], c[4], ws=self.ws,
                              stream=stream)
        else:
            fp4_quantize(self._cfg(3, step, round=FP4_ROUND_SR), dy, b["dy"], state=self.states[3], counters=c[3],
                         ws=self.ws, stream=stream)
            fp4_quantize(self._cfg(4, step, orient=FP4_ORIENT_COLWISE, rht=rht, round=FP4_ROUND_SR), dy, b["dyt"],
                         state=self.states[4], counters=c[4], ws=self.ws, stream=stream)
        _mark(mark, "dy/end")

    def _quantize_all_overlapped(self, x, w, dy, step, stream, mark=None):
        # side stream: the tensor amaxes of W, X and dY, the smallest tensor
        # first; main stream: the three quantized in the same order, each as
        # soon as its amax is ready, so only the smallest tensor's amax pass is
        # not hidden behind a conversion pass
        b, c, g, rht = self.bufs, self.counters, self.given, self.rht
        main = torch.cuda.current_stream() if stream is None else stream
        side = self.side
        self.ev_inputs.record(main)
        side.wait_event(self.ev_inputs)
        for t in (x, w, dy):
            t.record_stream(side)  # read on the side stream: keep the allocator from reusing it early
        w_cfg = dict(block=FP4_BLOCK_16x16)
        x_c = dict(orient=FP4_ORIENT_COLWISE, rht=rht)
        dy_r = dict(round=FP4_ROUND_SR)
        dy_c = dict(orient=FP4_ORIENT_COLWISE, rht=rht, round=FP4_ROUND_SR)
        giv = dict(tscale=FP4_TSCALE_GIVEN)
        jobs = [
            ("w", w.numel(),
             lambda: fp4_tensor_amax(self._cfg(2, step, **w_cfg), w, g[2], self.ws_side[0], stream=side),
             lambda: fp4_quantize(self._cfg(2, step, emit_transpose=True, **w_cfg, **giv), w, b["w"], b["wt"],
                                  state=g[2], counters=c[2], stream=main)),
            ("x", x.numel(),
             lambda: fp4_tensor_amax_dual(self._cfg(0, step), self._cfg(1, step, **x_c), x, g[0], g[1],
                                          self.ws_side[1], stream=side),
             lambda: fp4_quantize_dual(self._cfg(0, step, **giv), self._cfg(1, step, **x_c, **giv), x, b["x"],
                                       b["xt"], g[0], g[1], c[0], c[1], stream=main)),
            ("dy", dy.numel(),
             lambda: fp4_tensor_amax_dual(self._cfg(3, step, **dy_r), self._cfg(4, step, **dy_c), dy, g[3], g[4],
                                          self.ws_side[2], stream=side),
             lambda: fp4_quantize_dual(self._cfg(3, step, **dy_r, **giv), self._cfg(4, step, **dy_c, **giv), dy,
                                       b["dy"], b["dyt"], g[3], g[4], c[3], c[4], stream=main)),
        ]
        jobs.sort(key=lambda j: j[1])  # stable: W, X, dY among equal sizes
        for i, (_, _, amax, _) in enumerate(jobs):
            amax()
            self.ev_amax[i].record(side)
        for i, (name, _, _, quant) in enumerate(jobs):
            main.wait_event(self.ev_amax[i])
            _mark(mark, name)
            quant()
            _mark(mark, name + "/end")

    def gemms(self, y: torch.Tensor, dx: torch.Tensor, dw: torch.Tensor, stream=None, mark=None):
        """Fprop, Dgrad and Wgrad (`mark` as for quantize_all)."""
        b = self.bufs
        for name, (a_, b_), out in (("fprop", ("x", "w"), y), ("dgrad", ("dy", "wt"), dx),
                                    ("wgrad", ("dyt", "xt"), dw)):
            _mark(mark, name)
            if self.gemm_ws is not None:
                fp4_gemm(b[a_], b[b_], out, stream=stream, ws=self.gemm_ws)
            elif name == "fprop":
                fp4_linear_fprop(b[a_], b[b_], out, stream=stream)
            elif name == "dgrad":
                fp4_linear_dgrad(b[a_], b[b_], out, stream=stream)
            else:
                fp4_linear_wgrad(b[a_], b[b_], out, stream=stream)
            _mark(mark, name + "/end")

    def step(self, x, w, dy, y, dx, dw, step: int = 0, stream=None, mark=None):
        self.quantize_all(x, w, dy, step=step, stream=stream, mark=mark)
        self.gemms(y, dx, dw, stream=stream, mark=mark)

    def state_dict(self) -> dict:
        """The layer's only state across steps: the five held-amax records
        (held scaling), as host copies. Randomness is keyed by (seed, tensor id,
        step), which the caller passes in, so these records are all a resumed
        run needs to continue byte for byte."""
        return {"held_amax": [s.buf.cpu().clone() for s in self.states] if self.held else []}

    def load_state_dict(self, d: dict) -> None:
        recs = d["held_amax"]
        assert len(recs) == (5 if self.held else 0), "state does not match this layer's scaling mode"
        for s, r in zip(self.states, recs):
            s.buf.copy_(r)

    def step_host(self, x_h, w_h, dy_h, y_h, dx_h, dw_h, step: int = 0, stream=None):
        """`step` from pinned host tensors to pinned host tensors. The inputs are
        copied to device buffers on a host-to-device stream, the step runs on
        `stream` once they have landed, and the outputs are copied back on a
        device-to-host stream once it is done. The call returns at once. Two sets
        of device buffers alternate between calls, so one call's step runs while
        the next call's inputs come in and the previous call's outputs go out: a
        call's input copies wait only for the step two calls back to finish
        reading that set's inputs, and its step only for that step's output
        copies. `h2d_stream` can be made to wait on an event first; `ev_out` marks
        the end of the latest call's output copies (the copies run in order, so
        of all earlier ones too)."""
        dev = self.device
        if not hasattr(self, "h2d_stream"):
            self.h2d_stream = torch.cuda.Stream(device=dev)
            self.d2h_stream = torch.cuda.Stream(device=dev)
            self.host_slots = [
                {"in": {k: torch.empty(t.shape, dtype=t.dtype, device=dev)
                        for k, t in (("x", x_h), ("w", w_h), ("dy", dy_h))},
                 "out": {k: torch.empty(t.shape, dtype=t.dtype, device=dev)
                         for k, t in (("y", y_h), ("dx", dx_h), ("dw", dw_h))},
                 "ev_in": torch.cuda.Event(), "ev_done": torch.cuda.Event(), "ev_out": torch.cuda.Event()}
                for _ in range(2)]
            self.host_calls = 0
        main = torch.cuda.current_stream() if stream is None else stream
        slot = self.host_slots[self.host_calls % 2]
        self.host_calls += 1
        di, do = slot["in"], slot["out"]
        self.h2d_stream.wait_event(slot["ev_done"])  # the step two calls back has read these inputs
        with torch.cuda.stream(self.h2d_stream):
            for k, t in (("x", x_h), ("w", w_h), ("dy", dy_h)):
                di[k].copy_(t, non_blocking=True)
        slot["ev_in"].record(self.h2d_stream)
        main.wait_event(slot["ev_in"])
        main.wait_event(slot["ev_out"])  # ... and its output copies have read these outputs
        self.step(di["x"], di["w"], di["dy"], do["y"], do["dx"], do["dw"], step=step, stream=main)
        slot["ev_done"].record(main)
        self.d2h_stream.wait_event(slot["ev_done"])
        with torch.cuda.stream(self.d2h_stream):
            for k, t in (("y", y_h), ("dx", dx_h), ("dw", dw_h)):
                t.copy_(do[k], non_blocking=True)
        slot["ev_out"].record(self.d2h_stream)
        self.ev_out = slot["ev_out"]
