"""A resident sampler step: device buffers for one workload shape, and the two ways to
run it (inputs already on the device, or inputs copied from pinned host memory and
results copied back, all on one stream).

PyTorch only provides the memory and the stream; each step is one call of
dg_sampler_step in libdgsamp.
"""
from __future__ import annotations

import torch

from . import binding as B


class SamplerStep:
    """Owns the embedding table W (resident), the workspace and the outputs.  W is bf16, or
    with `scale` given an 8-bit table: W the E4M3 codes (uint8 [rows, d]) and `scale` the fp32
    row scales (from dg_quantize_e4m3, or the caller's own)."""

    def __init__(self, W: torch.Tensor, n_req: int, L_c: int, V: int, gamma: float,
                 vocab_start: int = 0, vocab_end: int | None = None, min_accept: int = 0,
                 device: str | torch.device = "cuda", scale: torch.Tensor | None = None,
                 two_pass: bool = False):
        self.device = torch.device(device)
        self.W = W
        self.scale = scale
        self.n_req, self.L_c, self.V = n_req, L_c, V
        self.R = n_req * L_c
        self.d = W.shape[1]
        self.gamma = float(gamma)
        self.vocab_start = vocab_start
        self.vocab_end = V if vocab_end is None else vocab_end
        self.min_accept = min_accept
        self.two_pass = bool(two_pass)  # statistics before the product (DG_STEP_TWO_PASS)
        R, d, dev = self.R, self.d, self.device
        self.out = {k: torch.empty(R, dtype=torch.float32, device=dev) for k in ("m", "lse", "H", "kappa")}
        self.out.update(argmax=torch.empty(R, dtype=torch.int32, device=dev),
                        order=torch.empty(R, dtype=torch.int32, device=dev),
                        mask=torch.empty(R, dtype=torch.uint8, device=dev),
                        n_accepted=torch.empty(n_req, dtype=torch.int32, device=dev),
                        E=torch.empty((R, d), dtype=torch.float32, device=dev))
        self.ws = (B.workspace_e4m3 if scale is not None else B.workspace)(
            R, max(1, self.vocab_end - self.vocab_start), d, dev)
        self.logits_dev = None
        self.budgets_dev = torch.empty(n_req, dtype=torch.float32, device=dev)

    # -- device-resident inputs
    def __call__(self, logits: torch.Tensor, budgets: torch.Tensor, stream=None) -> dict:
        if self.scale is not None:
            return B.dg_sampler_step_e4m3(logits, self.n_req, self.L_c, self.W, self.scale, self.gamma, budgets,
                                          min_accept=self.min_accept, vocab_start=self.vocab_start,
                                          vocab_end=self.vocab_end, V=self.V, out=self.out, ws=self.ws,
                                          stream=stream, two_pass=self.two_pass)
        return B.dg_sampler_step(logits, self.n_req, self.L_c, self.W, self.gamma, budgets,
                                 min_accept=self.min_accept, vocab_start=self.vocab_start,
                                 vocab_end=self.vocab_end, V=self.V, out=self.out, ws=self.ws,
                                 stream=stream, two_pass=self.two_pass)

    # -- host inputs and results
    def host_buffers(self, ldl: int | None = None) -> dict:
        """Pinned host tensors for the inputs and results of run_from_host()."""
        ldl = self.V if ldl is None else ldl
        h = {"logits": torch.empty((self.R, ldl), dtype=torch.float32, pin_memory=True),
             "budgets": torch.empty(self.n_req, dtype=torch.float32, pin_memory=True)}
        for k, v in self.out.items():
            h["out_" + k] = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
        if self.logits_dev is None or self.logits_dev.shape != h["logits"].shape:
            self.logits_dev = torch.empty(h["logits"].shape, dtype=torch.float32, device=self.device)
        return h

    def run_from_host(self, h: dict, stream=None) -> None:
        """H2D of logits and budgets, one step, D2H of every result; asynchronous on `stream`."""
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        with torch.cuda.stream(s):
            self.logits_dev.copy_(h["logits"], non_blocking=True)
            self.budgets_dev.copy_(h["budgets"], non_blocking=True)
            self(self.logits_dev, self.budgets_dev, stream=s)
            for k, v in self.out.items():
                h["out_" + k].copy_(v, non_blocking=True)

    def run_pipelined(self, h: dict, steps: int, stream=None) -> None:
        """`steps` steps from host buffers, the upload of each step's logits overlapping
        the previous step's kernels: two device logits buffers, uploads on a copy stream,
        kernels and the read-back of every step's results on `stream`, ordered by events."""
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        if not hasattr(self, "_copy_stream"):
            self._copy_stream = torch.cuda.Stream(device=self.device)
            self._bufs = [self.logits_dev, torch.empty_like(self.logits_dev)]
            self._budget_bufs = [self.budgets_dev, torch.empty_like(self.budgets_dev)]
        cs = self._copy_stream
        uploaded = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        cs.wait_stream(s)
        for t in range(steps):
            b = t & 1
            with torch.cuda.stream(cs):
                if t >= 2:
                    cs.wait_event(consumed[b])
                self._bufs[b].copy_(h["logits"], non_blocking=True)
                self._budget_bufs[b].copy_(h["budgets"], non_blocking=True)
                uploaded[b].record(cs)
            with torch.cuda.stream(s):
                s.wait_event(uploaded[b])
                self(self._bufs[b], self._budget_bufs[b], stream=s)
                consumed[b].record(s)
                for k, v in self.out.items():
                    h["out_" + k].copy_(v, non_blocking=True)
        s.wait_stream(cs)

    @staticmethod
    def h2d_bytes(h: dict) -> int:
        return h["logits"].numel() * 4 + h["budgets"].numel() * 4

    def d2h_bytes(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.out.values())


class SamplerLoop(SamplerStep):
    """A resident denoising loop: the step's buffers plus the loop state (canvas, eligible
    positions, previous argmax predictions, stable count, step count, converged flag) that
    each call of dg_sampler_loop_step reads and updates in place.  Successive calls on one
    stream, or a CUDA graph of several calls replayed, run successive steps.

    temperature 0 puts the argmax on the canvas; temperature > 0 draws the candidates
    (Philox key `seed`, counter offset advanced by one per call; a captured graph replays
    the offsets it was captured with)."""

    def __init__(self, W: torch.Tensor, n_req: int, L_c: int, V: int, gamma: float, stable_steps: int,
                 entropy_threshold: float, step_limit: int, temperature: float = 0.0, seed: int = 0, **kw):
        super().__init__(W, n_req, L_c, V, gamma, **kw)
        self.stable_steps = int(stable_steps)
        self.entropy_threshold = float(entropy_threshold)
        self.step_limit = int(step_limit)
        self.temperature = float(temperature)
        self.seed = int(seed)
        self.offset = 0
        if self.temperature != 0.0:
            self.out["candidate"] = torch.empty(self.R, dtype=torch.int32, device=self.device)
        self.state = B.new_loop_state(n_req, L_c, self.device)

    def reset(self, canvas0: torch.Tensor | None = None) -> None:
        """Back to the starting state (in place, so captured graphs stay valid)."""
        if canvas0 is None:
            self.state["canvas"].zero_()
        else:
            self.state["canvas"].copy_(canvas0.reshape(-1))
        self.state["eligible"].fill_(1)
        self.state["prev_argmax"].fill_(-1)
        for k in ("stable", "steps", "converged"):
            self.state[k].zero_()
        self.offset = 0

    def __call__(self, logits: torch.Tensor, budgets: torch.Tensor, stream=None) -> dict:
        if self.scale is not None:
            o = B.dg_sampler_loop_step_e4m3(logits, self.n_req, self.L_c, self.W, self.scale, self.gamma, budgets,
                                            self.state, self.stable_steps, self.entropy_threshold,
                                            self.step_limit, min_accept=self.min_accept,
                                            vocab_start=self.vocab_start, vocab_end=self.vocab_end, V=self.V,
                                            out=self.out, ws=self.ws, temperature=self.temperature,
                                            seed=self.seed, offset=self.offset, stream=stream,
                                            two_pass=self.two_pass)
            self.offset += 1
            return o
        o = B.dg_sampler_loop_step(logits, self.n_req, self.L_c, self.W, self.gamma, budgets, self.state,
                                   self.stable_steps, self.entropy_threshold, self.step_limit,
                                   min_accept=self.min_accept, vocab_start=self.vocab_start,
                                   vocab_end=self.vocab_end, V=self.V, out=self.out, ws=self.ws,
                                   temperature=self.temperature, seed=self.seed, offset=self.offset,
                                   stream=stream, two_pass=self.two_pass)
        self.offset += 1
        return o
