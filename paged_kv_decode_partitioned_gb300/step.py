"""A decode step with its buffers allocated once: the way a serving loop calls the library.

``DecodeStep`` binds the inputs of one batch (device tensors), picks the
entry points for a mode and owns the output, the partial buffers and the
workspace, so that repeated calls launch kernels and nothing else.

Modes (page: project_6 commit cd0d9e1, "qwen3_6_scripts": the forward_decode
heuristic and the V2 description):

* ``"single"``      -- ``pa_decode``: every sequence in one pass (V1);
* ``"partitioned"`` -- ``pa_decode_partitioned`` then ``pa_partition_reduce``
  with one partition size for every sequence (V2, phase 1 + phase 2);
* ``"auto"``        -- ``pa_decode_auto``: sequences up to
  ``single_pass_max_len`` tokens in one pass, longer ones partitioned and
  merged; the library picks the launch form (single-pass grid, dense
  partitioned grid + reduce, or the device work list) and, when asked
  (``single_pass_max_len=-1``, ``partition_size=0``), the threshold and the
  partition size.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (AUTO_DENSE, AUTO_SINGLE_PASS, PHASE_ATTEND, PHASE_PLAN, PHASE_REDUCE,
               auto_resolve, auto_workspace_bytes, decode, decode_auto, decode_partitioned,
               num_partitions, partition_buffers, partition_reduce)

MODES = ("single", "partitioned", "auto")


class DecodeStep:
    def __init__(self, mode: str, query, key_cache, value_cache, block_tables, seq_lens,
                 scale: float, *, max_seq_len: int, partition_size: int = 512,
                 single_pass_max_len: int = 8192, out: Optional[torch.Tensor] = None,
                 max_total_tokens: int = 0):
        if mode not in MODES:
            raise ValueError(f"mode must be one of {MODES}")
        self.mode = mode
        self.query, self.key_cache, self.value_cache = query, key_cache, value_cache
        self.block_tables, self.seq_lens = block_tables, seq_lens
        self.scale = float(scale)
        self.max_seq_len = int(max_seq_len)
        self.partition_size = int(partition_size)
        self.single_pass_max_len = int(single_pass_max_len)
        self.out = torch.empty_like(query) if out is None else out
        S, Hq, D = query.shape
        Hkv = key_cache.shape[2]
        dev = query.device
        self.tmp_out = self.exp_sums = self.max_logits = self.workspace = None
        self.max_total_tokens = int(max_total_tokens)
        if mode == "partitioned":
            self.max_num_partitions = max(1, num_partitions(self.max_seq_len, partition_size))
            self.tmp_out, self.exp_sums, self.max_logits = partition_buffers(
                S, Hq, D, self.max_num_partitions, dev)
        elif mode == "auto":
            bs = key_cache.shape[1]
            with torch.cuda.device(dev):
                self.resolved = auto_resolve(S, Hkv, D, bs, self.max_seq_len,
                                             self.single_pass_max_len, self.partition_size,
                                             max_total_tokens=self.max_total_tokens)
                need = auto_workspace_bytes(S, Hq, Hkv, D, bs, self.max_seq_len,
                                            self.max_total_tokens, self.single_pass_max_len,
                                            self.partition_size)
            self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

    @property
    def form(self) -> Optional[int]:
        """The launch form ``pa_decode_auto`` takes (auto mode; AUTO_* of the binding)."""
        return self.resolved[2] if self.mode == "auto" else None

    @property
    def kernels_per_call(self) -> int:
        """Kernel launches one call makes (single: 1; partitioned: 2; auto: 1, 2 or 3 by
        the resolved launch form)."""
        if self.mode == "single":
            return 1
        if self.mode == "partitioned":
            return 2
        return {AUTO_SINGLE_PASS: 1, AUTO_DENSE: 2}.get(self.form, 3)

    @property
    def attention_kernel(self) -> str:
        """Name of the kernel that reads the KV cache (the step's dominant kernel)."""
        if self.mode == "auto":
            return {AUTO_SINGLE_PASS: "pa_attn_kernel<single>",
                    AUTO_DENSE: "pa_attn_kernel<partitioned>"}.get(
                        self.form, "pa_attn_kernel<worklist>")
        return {"single": "pa_attn_kernel<single>",
                "partitioned": "pa_attn_kernel<partitioned>"}[self.mode]

    def launches(self):
        """The step as (label, callable) pairs in launch order, one kernel each.

        Running them in order on one stream is exactly one ``__call__``; a
        caller can record stream events between them to time one kernel.
        The attention kernel's label is ``"attention"``.
        """
        if self.mode == "single":
            return [("attention", self.__call__)]
        if self.mode == "partitioned":
            def attend():
                decode_partitioned(self.query, self.key_cache, self.value_cache,
                                   self.block_tables, self.seq_lens, self.scale,
                                   self.partition_size, self.max_num_partitions, self.tmp_out,
                                   self.exp_sums, self.max_logits)

            def reduce():
                partition_reduce(self.tmp_out, self.exp_sums, self.max_logits, self.seq_lens,
                                 self.partition_size, out=self.out, dtype=self.out.dtype)
            return [("attention", attend), ("reduce", reduce)]

        def phase(mask):
            return lambda: decode_auto(self.query, self.key_cache, self.value_cache,
                                       self.block_tables, self.seq_lens, self.scale,
                                       self.max_seq_len, self.single_pass_max_len,
                                       self.partition_size, workspace=self.workspace,
                                       out=self.out, phases=mask,
                                       max_total_tokens=self.max_total_tokens)
        if self.form == AUTO_SINGLE_PASS:   # one single-pass launch
            return [("attention", phase(PHASE_PLAN | PHASE_ATTEND | PHASE_REDUCE))]
        if self.form == AUTO_DENSE:          # partitioned grid, then the dense reduce
            return [("attention", phase(PHASE_ATTEND)), ("reduce", phase(PHASE_REDUCE))]
        return [("plan", phase(PHASE_PLAN)), ("attention", phase(PHASE_ATTEND)),
                ("reduce", phase(PHASE_REDUCE))]

    def __call__(self) -> torch.Tensor:
        if self.mode == "single":
            return decode(self.query, self.key_cache, self.value_cache, self.block_tables,
                          self.seq_lens, self.scale, out=self.out)
        if self.mode == "partitioned":
            decode_partitioned(self.query, self.key_cache, self.value_cache, self.block_tables,
                               self.seq_lens, self.scale, self.partition_size,
                               self.max_num_partitions, self.tmp_out, self.exp_sums,
                               self.max_logits)
            return partition_reduce(self.tmp_out, self.exp_sums, self.max_logits, self.seq_lens,
                                    self.partition_size, out=self.out, dtype=self.out.dtype)
        return decode_auto(self.query, self.key_cache, self.value_cache, self.block_tables,
                           self.seq_lens, self.scale, self.max_seq_len,
                           self.single_pass_max_len, self.partition_size,
                           workspace=self.workspace, out=self.out,
                           max_total_tokens=self.max_total_tokens)
