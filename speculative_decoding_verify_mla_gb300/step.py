"""One whole verify step (attention + greedy verify) on preallocated buffers."""
from __future__ import annotations

import torch

from . import binding as B


class VerifyStep:
    """Runs mla_verify_decode and spec_verify_greedy for one batch.

    The two parts are independent (the greedy verify reads the target logits,
    not the attention output), so the greedy kernel runs on a side stream
    forked from and joined back into the caller's stream: the step costs
    about max(attention, greedy) instead of their sum.  Output buffers and
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
        self.accepted = torch.empty(R, dtype=torch.int32, device=device)
        self.next_tokens = torch.empty(R, dtype=torch.int32, device=device)
        self.kv_lens_out = torch.empty(R, dtype=torch.int32, device=device)
        self.side = torch.cuda.Stream(device=device)

    def __call__(self, q_latent, kv_pages, block_table, kv_bounds, gate, softmax_scale,
                 logits, draft_tokens, kv_lens_in):
        main = torch.cuda.current_stream(self.device)
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            B.spec_verify_greedy(logits, draft_tokens, kv_lens_in, self.k,
                                 workspace=self.greedy_ws, argmax_ids=self.argmax,
                                 accepted=self.accepted, next_tokens=self.next_tokens,
                                 kv_lens_out=self.kv_lens_out)
        B.mla_verify_decode(q_latent, kv_pages, block_table, kv_bounds, gate, self.k + 1,
                            softmax_scale, num_splits=self.num_splits, workspace=self.attn_ws,
                            out=self.out, lse=self.lse, status=self.status)
        main.wait_stream(self.side)
        return self.out, self.lse, self.argmax, self.accepted, self.next_tokens, self.kv_lens_out

    @property
    def attention_launches(self) -> int:
        """Kernels one mla_verify_decode call enqueues: the balanced plan adds a
        plan kernel and the merge; uniform splits add the merge when S > 1."""
        if self.num_splits == B.SV_SPLITS_BALANCED:
            return 3
        return 1 + (1 if self.num_splits > 1 else 0)

    @property
    def launches_per_step(self) -> int:
        """Kernels one step enqueues: the attention call's kernels + greedy."""
        return self.attention_launches + 1
