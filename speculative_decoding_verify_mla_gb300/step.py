"""One whole verify step (attention + greedy verify) on preallocated buffers."""
from __future__ import annotations

import torch

from . import binding as B


class VerifyStep:
    """Runs mla_verify_decode and spec_verify_greedy for one batch.

    The two parts are independent (the greedy verify reads the target logits,
    not the attention output), so the greedy kernel runs on a side stream
    forked from and joined back into the caller's stream: the step costs
    about max(attention, greedy) instead of their sum.  The attention is
    enqueued first so that its grid (one CTA per SM, nearly all of the SM's
    shared memory) is placed before the greedy CTAs fill the SMs; a CUDA
    graph captured from the step keeps that order (captured greedy-first,
    the C = 32 step replayed in 118.9 us instead of 104.9 us on GB300).  Output buffers and
    both workspaces are allocated once (torch) and reused, so a step enqueues
    exactly the library's kernels and nothing else."""

    def __init__(self, device, R: int, k: int, H: int, V: int, max_pages: int,
                 num_splits: int = 0):
        device = torch.device(device)
        self.device = device
        self.R, self.k, self.H, self.V = R, k, H, V
        self.T = R * (k + 1)
        self.max_pages = max_pages
        self.num_splits = num_splits or B.num_splits_for(R, k + 1, H, max_pages)
        T = self.T
        self.out = torch.empty((T, H, B.SV_LATENT_DIM), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        ws = B.attention_workspace_bytes(T, H, self.num_splits)
        self.attn_ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=device)
        self.greedy_ws = torch.zeros(B.greedy_workspace_bytes(T, V), dtype=torch.uint8,
                                     device=device)
        self.argmax = torch.empty(T, dtype=torch.int32, device=device)
        # the per-request results are rows of one [3, R] block, so a caller
        # reads all of them back with a single device-to-host copy
        self.results = torch.empty((3, R), dtype=torch.int32, device=device)
        self.accepted, self.next_tokens, self.kv_lens_out = self.results[0], self.results[1], self.results[2]
        self.side = torch.cuda.Stream(device=device)

    def __call__(self, q_latent, kv_pages, block_table, kv_bounds, gate, softmax_scale,
                 logits, draft_tokens, kv_lens_in):
        main = torch.cuda.current_stream(self.device)
        self.side.wait_stream(main)
        B.mla_verify_decode(q_latent, kv_pages, block_table, kv_bounds, gate, self.k + 1,
                            softmax_scale, num_splits=self.num_splits, workspace=self.attn_ws,
                            out=self.out, lse=self.lse, status=self.status)
        with torch.cuda.stream(self.side):
            B.spec_verify_greedy(logits, draft_tokens, kv_lens_in, self.k,
                                 workspace=self.greedy_ws, argmax_ids=self.argmax,
                                 accepted=self.accepted, next_tokens=self.next_tokens,
                                 kv_lens_out=self.kv_lens_out)
        main.wait_stream(self.side)
        return self.out, self.lse, self.argmax, self.accepted, self.next_tokens, self.kv_lens_out

    def run_staged(self, att, ver, kv_pages, softmax_scale):
        """The step fed from host memory through two StagedInputs: ``att``
        (q_latent, gate, block_table, kv_bounds) is uploaded on the caller's
        stream ahead of the attention, ``ver`` (logits, draft_tokens,
        kv_lens_in) on the side stream ahead of the greedy verify, so the
        logits copy overlaps the attention.  The logits copy starts only once
        the attention inputs have landed: both copies share the host-to-device
        bandwidth, and the attention waits for its inputs while the greedy
        verify, much shorter, can wait for the logits.  Returns the [3, R]
        results block (accepted, next_tokens, kv_lens_out) on the caller's
        stream."""
        main = torch.cuda.current_stream(self.device)
        att.upload()  # the small attention inputs first, so the attention can start
        self.side.wait_stream(main)  # ... alone on the link
        with torch.cuda.stream(self.side):
            ver.upload()  # the logits copy overlaps the attention
        B.mla_verify_decode(att.dev["q_latent"], kv_pages, att.dev["block_table"], att.dev["kv_bounds"],
                            att.dev["gate"], self.k + 1, softmax_scale, num_splits=self.num_splits,
                            workspace=self.attn_ws, out=self.out, lse=self.lse, status=self.status)
        with torch.cuda.stream(self.side):
            B.spec_verify_greedy(ver.dev["logits"], ver.dev["draft_tokens"], ver.dev["kv_lens_in"], self.k,
                                 workspace=self.greedy_ws, argmax_ids=self.argmax,
                                 accepted=self.accepted, next_tokens=self.next_tokens,
                                 kv_lens_out=self.kv_lens_out)
        main.wait_stream(self.side)
        return self.results

    @property
    def attention_launches(self) -> int:
        """Kernels one mla_verify_decode call enqueues: the balanced plan adds a
        plan kernel and the merge; the wave mode and uniform splits (S > 1) add
        the merge."""
        if self.num_splits == B.SV_SPLITS_BALANCED:
            return 3
        if self.num_splits == B.SV_SPLITS_WAVE:
            return 2
        return 1 + (1 if self.num_splits > 1 else 0)

    @property
    def launches_per_step(self) -> int:
        """Kernels one step enqueues: the attention call's kernels + greedy."""
        return self.attention_launches + 1


class StagedInputs:
    """A step's inputs in one pinned host buffer mirrored by one device buffer
    (each tensor 256-byte aligned inside), so that a step moves all its
    inputs with a single host-to-device copy instead of one per tensor.

    ``specs`` maps a name to (shape, dtype).  Fill ``host[name]`` (pinned
    views), call ``upload()`` on the step's stream, and pass ``dev[name]``
    (device views) to the step."""

    def __init__(self, device, specs: dict):
        device = torch.device(device)
        offsets, off = {}, 0
        for name, (shape, dtype) in specs.items():
            nbytes = int(torch.Size(shape).numel()) * torch.tensor([], dtype=dtype).element_size()
            offsets[name] = (off, nbytes, tuple(shape), dtype)
            off += (nbytes + 255) // 256 * 256
        self.nbytes = off
        self._host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self._dev = torch.empty(off, dtype=torch.uint8, device=device)
        self.host, self.dev = {}, {}
        for name, (o, n, shape, dtype) in offsets.items():
            self.host[name] = self._host[o:o + n].view(dtype).view(shape)
            self.dev[name] = self._dev[o:o + n].view(dtype).view(shape)

    def upload(self):
        """Host -> device copy of every input, asynchronous on the current stream."""
        self._dev.copy_(self._host, non_blocking=True)
