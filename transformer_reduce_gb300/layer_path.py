"""One pass of the reduce hot path of a Transformer layer, through the C ABI.

A pre-LayerNorm encoder layer touches the five kernels in this order on one
stream (forward, then backward in reverse):

    LN1 fw -> softmax fw -> LN2 fw -> LN2 bw (dinp, dgamma/dbeta)
           -> softmax bw -> LN1 bw (dinp, dgamma/dbeta)

``LayerReducePath`` owns the device buffers of one such pass (inputs drawn by
``workloads``, outputs, the dgamma/dbeta workspaces) and issues the calls.
Every call goes through ``_lib`` (raw pointers, the caller's stream); torch is
used only to hold device and pinned host memory and to copy between them.
"""
from __future__ import annotations

import dataclasses

import torch

from . import _lib, traffic, workloads

_DT = {"f32": _lib.LS_F32, "f16": _lib.LS_F16, "bf16": _lib.LS_BF16}


def _ok(status, where):
    if status != _lib.LS_OK:
        raise _lib.LsError(status, where)


@dataclasses.dataclass
class _LnBuffers:
    case: workloads.LayerNormCase
    x: torch.Tensor
    gamma: torch.Tensor
    beta: torch.Tensor
    dy: torch.Tensor
    y: torch.Tensor
    mean: torch.Tensor
    rstd: torch.Tensor
    dx: torch.Tensor
    dgamma: torch.Tensor
    dbeta: torch.Tensor
    ws: torch.Tensor
    ws_fused: torch.Tensor


class LayerReducePath:
    def __init__(self, softmax_case: workloads.SoftmaxCase, ln_cases, device="cuda"):
        self.device = torch.device(device)
        self.sm = softmax_case
        si = workloads.softmax_inputs(softmax_case, device=self.device)
        self.lengths = si["lengths"]
        self.scores, self.mask, self.dprobs = si["scores"], si["mask"], si["dout"]
        self.probs = torch.empty_like(self.scores)
        self.dscores = torch.empty_like(self.scores)
        self.ln = []
        for case in ln_cases:
            li = workloads.layernorm_inputs(case, device=self.device)
            n = _lib.ls_layernorm_bw_dgamma_dbeta_workspace_size(case.rows, case.hidden)
            nf = _lib.ls_layernorm_bw_workspace_size(case.rows, case.hidden)
            f32 = dict(device=self.device, dtype=torch.float32)
            self.ln.append(_LnBuffers(
                case=case, x=li["x"], gamma=li["gamma"], beta=li["beta"], dy=li["dy"],
                y=torch.empty_like(li["x"]), mean=torch.empty(case.rows, **f32),
                rstd=torch.empty(case.rows, **f32), dx=torch.empty_like(li["x"]),
                dgamma=torch.empty(case.hidden, **f32), dbeta=torch.empty(case.hidden, **f32),
                ws=torch.empty(max(n, 16) // 4, **f32),
                ws_fused=torch.empty(max(nf, 16) // 4, **f32)))
        self._host = None

    # ---- the hot path ------------------------------------------------------
    def _ln_fw(self, b: _LnBuffers, st):
        c = b.case
        _ok(_lib.ls_layernorm_fw(b.y.data_ptr(), b.mean.data_ptr(), b.rstd.data_ptr(),
                                 b.x.data_ptr(), b.gamma.data_ptr(), b.beta.data_ptr(),
                                 c.rows, c.hidden, c.eps, _DT[c.dtype], st), "ls_layernorm_fw")

    def _ln_dinp(self, b: _LnBuffers, st):
        c = b.case
        _ok(_lib.ls_layernorm_bw_dinp(b.dx.data_ptr(), b.dy.data_ptr(), b.x.data_ptr(),
                                      b.gamma.data_ptr(), b.mean.data_ptr(), b.rstd.data_ptr(),
                                      c.rows, c.hidden, _DT[c.dtype], st), "ls_layernorm_bw_dinp")

    def _ln_dgdb(self, b: _LnBuffers, st):
        c = b.case
        _ok(_lib.ls_layernorm_bw_dgamma_dbeta(
            b.dgamma.data_ptr(), b.dbeta.data_ptr(), b.dy.data_ptr(), b.x.data_ptr(),
            b.mean.data_ptr(), b.rstd.data_ptr(), c.rows, c.hidden, b.ws.data_ptr(),
            b.ws.numel() * 4, _DT[c.dtype], st), "ls_layernorm_bw_dgamma_dbeta")

    def _ln_bw_fused(self, b: _LnBuffers, st):
        c = b.case
        _ok(_lib.ls_layernorm_bw(
            b.dx.data_ptr(), b.dgamma.data_ptr(), b.dbeta.data_ptr(), b.dy.data_ptr(),
            b.x.data_ptr(), b.gamma.data_ptr(), b.mean.data_ptr(), b.rstd.data_ptr(), c.rows,
            c.hidden, b.ws_fused.data_ptr(), b.ws_fused.numel() * 4, _DT[c.dtype], st),
            "ls_layernorm_bw")

    def _softmax_bw_masked(self, st):
        s = self.sm
        _ok(_lib.ls_softmax_bw_masked(
            self.dscores.data_ptr(), self.dprobs.data_ptr(), self.probs.data_ptr(),
            0 if self.mask is None else self.mask.data_ptr(), s.B, s.H, s.T, s.T, s.causal,
            _DT[s.dtype], st), "ls_softmax_bw_masked")

    def _softmax_fw(self, st):
        s = self.sm
        _ok(_lib.ls_softmax_fw(self.probs.data_ptr(), self.scores.data_ptr(),
                               0 if self.mask is None else self.mask.data_ptr(),
                               s.B, s.H, s.T, s.T, s.causal, _DT[s.dtype], st), "ls_softmax_fw")

    def _softmax_bw(self, st):
        s = self.sm
        _ok(_lib.ls_softmax_bw(self.dscores.data_ptr(), self.dprobs.data_ptr(),
                               self.probs.data_ptr(), s.B, s.H, s.T, s.T, _DT[s.dtype], st),
            "ls_softmax_bw")

    def sequence(self):
        """The (name, call(stream_handle)) list of one pass, in stream order."""
        ln1 = self.ln[0]
        ln2 = self.ln[1] if len(self.ln) > 1 else None
        seq = [("ln_fw", lambda st: self._ln_fw(ln1, st)),
               ("softmax_fw", self._softmax_fw)]
        if ln2 is not None:
            seq += [("ln_fw", lambda st: self._ln_fw(ln2, st)),
                    ("ln_dinp", lambda st: self._ln_dinp(ln2, st)),
                    ("ln_dgdb", lambda st: self._ln_dgdb(ln2, st))]
        seq += [("softmax_bw", self._softmax_bw),
                ("ln_dinp", lambda st: self._ln_dinp(ln1, st)),
                ("ln_dgdb", lambda st: self._ln_dgdb(ln1, st))]
        return seq

    def fused_sequence(self):
        """The same layer with the fused LayerNorm backward (dx, dgamma and
        dbeta from one read of dy and x) and the softmax backward that takes
        the mask and reads only visible keys; (name, call) in stream order."""
        ln1 = self.ln[0]
        ln2 = self.ln[1] if len(self.ln) > 1 else None
        seq = [("ln_fw", lambda st: self._ln_fw(ln1, st)),
               ("softmax_fw", self._softmax_fw)]
        if ln2 is not None:
            seq += [("ln_fw", lambda st: self._ln_fw(ln2, st)),
                    ("ln_bw", lambda st: self._ln_bw_fused(ln2, st))]
        seq += [("softmax_bw_masked", self._softmax_bw_masked),
                ("ln_bw", lambda st: self._ln_bw_fused(ln1, st))]
        return seq

    def run_fused(self, stream=None, timers=None):
        """Enqueue one pass of fused_sequence() on one stream (timers as in
        run()).  Same outputs as run(), up to the rounding of the fused
        kernels' own summation order."""
        self._enqueue(self.fused_sequence(), stream, timers)

    def run(self, stream=None, timers=None):
        """Enqueue one pass on `stream` (default: torch's current stream).
        timers: optional dict name -> list; a (start, end) CUDA event pair
        recorded on the same stream is appended around each call."""
        self._enqueue(self.sequence(), stream, timers)

    def _enqueue(self, seq, stream, timers):
        stream = stream or torch.cuda.current_stream(self.device)
        st = stream.cuda_stream
        for name, call in seq:
            if timers is None:
                call(st)
                continue
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call(st)
            e1.record(stream)
            timers.setdefault(name, []).append((e0, e1))

    def run_overlapped(self, stream, side):
        """One pass with the gamma/beta gradients on a second stream.

        Nothing later in a layer's backward reads dgamma / dbeta (they are
        parameter gradients), so each LayerNorm's dgamma/dbeta call runs on
        `side` beside the rest of the backward on `stream`, but no earlier
        than a real layer could issue it:

        * LN2's dy (the gradient arriving from the block above) exists when
          the backward starts, so LN2's dgamma/dbeta starts once the forward
          statistics exist and overlaps LN2's input gradient and the softmax
          backward;
        * LN1's dy is the attention block's input gradient, which exists only
          after the softmax backward, so LN1's dgamma/dbeta waits for an event
          recorded after the softmax backward and overlaps only LN1's own
          input gradient.

        The pass ends with `stream` waiting for `side`, so the next pass
        (which rewrites the statistics) starts after both.  Same calls and
        results as run(); only the order between independent calls differs."""
        st, sd = stream.cuda_stream, side.cuda_stream
        ln1 = self.ln[0]
        ln2 = self.ln[1] if len(self.ln) > 1 else None
        self._ln_fw(ln1, st)
        self._softmax_fw(st)
        if ln2 is not None:
            self._ln_fw(ln2, st)
            fw_done = torch.cuda.Event()
            fw_done.record(stream)
            side.wait_event(fw_done)
            self._ln_dgdb(ln2, sd)
            self._ln_dinp(ln2, st)
        self._softmax_bw(st)
        dy1_ready = torch.cuda.Event()
        dy1_ready.record(stream)
        side.wait_event(dy1_ready)
        self._ln_dgdb(ln1, sd)
        self._ln_dinp(ln1, st)
        side_done = torch.cuda.Event()
        side_done.record(side)
        stream.wait_event(side_done)

    # ---- accounting ----------------------------------------------------------
    def kernel_bytes(self) -> dict:
        """Algorithmic bytes of each call of one pass (name -> list of bytes)."""
        s = self.sm
        out = {}
        for name, _ in self.sequence():
            out.setdefault(name, [])
        out["softmax_fw"].append(traffic.softmax_fw_bytes(s.B, s.H, s.T, self.lengths, s.causal,
                                                          s.dtype, self.mask is not None))
        out["softmax_bw"].append(traffic.softmax_bw_bytes(s.B, s.H, s.T, s.dtype))
        for b in self.ln:
            c = b.case
            out["ln_fw"].append(traffic.layernorm_fw_bytes(c.rows, c.hidden, c.dtype))
            out["ln_dinp"].append(traffic.layernorm_dinp_bytes(c.rows, c.hidden, c.dtype))
            out["ln_dgdb"].append(traffic.layernorm_dgdb_bytes(c.rows, c.hidden, c.dtype))
        return out

    def step_bytes(self) -> int:
        return sum(sum(v) for v in self.kernel_bytes().values())

    def fused_kernel_bytes(self) -> dict:
        """Algorithmic bytes of each call of one fused_sequence() pass."""
        s = self.sm
        kb = self.kernel_bytes()
        out = {"ln_fw": kb["ln_fw"], "softmax_fw": kb["softmax_fw"], "ln_bw": [],
               "softmax_bw_masked": [traffic.softmax_bw_masked_bytes(
                   s.B, s.H, s.T, self.lengths, s.causal, s.dtype, self.mask is not None)]}
        for b in self.ln:
            c = b.case
            out["ln_bw"].append(traffic.layernorm_bw_fused_bytes(c.rows, c.hidden, c.dtype))
        return out

    def fused_step_bytes(self) -> int:
        return sum(sum(v) for v in self.fused_kernel_bytes().values())

    def dense_step_bytes(self) -> int:
        """Bytes of one pass if the softmax forward read every key (no
        masked-key skipping): the dense-equivalent count."""
        s = self.sm
        skipped = (traffic.softmax_fw_bytes(s.B, s.H, s.T, [s.T] * s.B, False, s.dtype,
                                            self.mask is not None)
                   - traffic.softmax_fw_bytes(s.B, s.H, s.T, self.lengths, s.causal, s.dtype,
                                              self.mask is not None))
        return self.step_bytes() + skipped

    def rows(self) -> dict:
        return {"softmax_rows": 2 * self.sm.rows,  # forward and backward
                "layernorm_rows": sum(3 * b.case.rows for b in self.ln)}

    # ---- end-to-end copies -----------------------------------------------------
    def _inputs(self):
        t = [self.scores, self.dprobs] + ([self.mask] if self.mask is not None else [])
        for b in self.ln:
            t += [b.x, b.gamma, b.beta, b.dy]
        return t

    def _outputs(self):
        t = [self.probs, self.dscores]
        for b in self.ln:
            t += [b.y, b.mean, b.rstd, b.dx, b.dgamma, b.dbeta]
        return t

    def host_buffers(self):
        """Pinned host copies of every input and output of a pass."""
        if self._host is None:
            self._host = ([x.cpu().pin_memory() for x in self._inputs()],
                          [torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
                           for x in self._outputs()])
        return self._host

    def h2d_bytes(self) -> int:
        return sum(x.numel() * x.element_size() for x in self._inputs())

    def d2h_bytes(self) -> int:
        return sum(x.numel() * x.element_size() for x in self._outputs())

    def upload(self, stream):
        hin, _ = self.host_buffers()
        with torch.cuda.stream(stream):
            for d, h in zip(self._inputs(), hin):
                d.copy_(h, non_blocking=True)

    def download(self, stream):
        _, hout = self.host_buffers()
        with torch.cuda.stream(stream):
            for h, d in zip(hout, self._outputs()):
                h.copy_(d, non_blocking=True)


class PipelinedPasses:
    """Passes fed from pinned host memory with the copies overlapped.

    Two device copies of the pass's buffers (``paths[0]`` and ``paths[1]``);
    step k uses copy k % 2 (its kernels one after the other on one stream, as
    ``run`` issues them).  The host-to-device copies, the kernels and the
    device-to-host copies run on their own streams; each copy direction can
    be split over ``lanes`` streams (tensors dealt out largest first), but one
    stream per direction measured fastest on GB300 (4.09 ms per step against
    4.13 with two and 4.15 with four).  Events order step k's upload after
    step k-2's kernels (they read the same input buffers), its kernels after
    its upload and after step k-2's download (the same output buffers), and
    its download after its kernels.  In steady state both copy directions and
    the kernels of neighbouring steps run at the same time.  Every step
    uploads every input from the same pinned host buffers and downloads every
    output into one set of pinned host buffers."""

    def __init__(self, paths, lanes: int = 1):
        assert len(paths) == 2
        self.paths = paths
        self.dev = paths[0].device
        self.hin, self.hout = paths[0].host_buffers()
        self.s_up = [torch.cuda.Stream(self.dev) for _ in range(lanes)]
        self.s_run = torch.cuda.Stream(self.dev)
        self.s_down = [torch.cuda.Stream(self.dev) for _ in range(lanes)]
        self.in_lane = self._deal([h.numel() * h.element_size() for h in self.hin], lanes)
        self.out_lane = self._deal([h.numel() * h.element_size() for h in self.hout], lanes)

    @staticmethod
    def _deal(sizes, lanes):
        load = [0] * lanes
        lane_of = [0] * len(sizes)
        for i in sorted(range(len(sizes)), key=lambda i: -sizes[i]):
            j = min(range(lanes), key=lambda j: load[j])
            lane_of[i] = j
            load[j] += sizes[i]
        return lane_of

    def _copies(self, streams, lane_of, pairs):
        done = []
        for j, st in enumerate(streams):
            with torch.cuda.stream(st):
                for i, (dst, src) in enumerate(pairs):
                    if lane_of[i] == j:
                        dst.copy_(src, non_blocking=True)
            e = torch.cuda.Event()
            e.record(st)
            done.append(e)
        return done

    def run(self, steps: int):
        """Enqueue `steps` passes; returns (start, end) CUDA events around all
        of them."""
        up, comp, down = [], [], []
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(self.s_run)
        for st in self.s_up + self.s_down:
            st.wait_event(start)
        for k in range(steps):
            p = self.paths[k % 2]
            if k >= 2:
                for st in self.s_up:
                    st.wait_event(comp[k - 2])
            up.append(self._copies(self.s_up, self.in_lane, list(zip(p._inputs(), self.hin))))
            for e in up[k]:
                self.s_run.wait_event(e)
            if k >= 2:
                for e in down[k - 2]:
                    self.s_run.wait_event(e)
            p.run(self.s_run)
            comp.append(torch.cuda.Event())
            comp[k].record(self.s_run)
            for st in self.s_down:
                st.wait_event(comp[k])
            down.append(self._copies(self.s_down, self.out_lane,
                                     list(zip(self.hout, p._outputs()))))
        # the end waits for every stream's last work
        for e in down[-1]:
            self.s_run.wait_event(e)
        end.record(self.s_run)
        return start, end
