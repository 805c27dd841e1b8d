"""One DSA attention layer's decode state: the two paged caches and the calls of a decode
step, on one CUDA device.  Plumbing only -- torch allocates the memory and every
computation is a call into the C ABI.
"""

import torch

from . import (alloc_k_cache, alloc_kv_cache, quant_kv_mxfp8, quant_kv_fp8, decode_step, indexer_topk,
               sparse_attn, sparse_attn_workspace_size)


class DsaDecodeLayer:
    """Paged MXFP8 indexer K-cache + paged FP8 latent cache of ``num_pages`` 64-token pages.

    A decode step writes the step's new tokens into both caches, runs the fused indexer +
    Top-K, then sparse attention over the selected entries.
    """

    def __init__(self, num_pages, h_i, h_s, topk, sm_scale, device="cuda"):
        self.device = torch.device(device)
        self.num_pages = int(num_pages)
        self.h_i, self.h_s, self.topk, self.sm_scale = h_i, h_s, topk, float(sm_scale)
        self.k_cache = alloc_k_cache(num_pages, self.device)
        self.kv_cache = alloc_kv_cache(num_pages, self.device)
        self._ws = {}
        self._bufs = {}

    def write(self, k, kv, slot_mapping):
        """Quantise and store new tokens: k bf16 [n, 128], kv bf16 [n, 576], slots int64 [n]."""
        quant_kv_mxfp8(k, slot_mapping, self.k_cache)
        quant_kv_fp8(kv, slot_mapping, self.kv_cache)

    def _buffers(self, n_q):
        b = self._bufs.get(n_q)
        if b is None:
            dev = self.device
            b = {
                "idx": torch.empty(n_q, self.topk, dtype=torch.int32, device=dev),
                "out": torch.empty(n_q, self.h_s, 512, dtype=torch.bfloat16, device=dev),
                "lse": torch.empty(n_q, self.h_s, dtype=torch.float32, device=dev),
            }
            ws = sparse_attn_workspace_size(n_q, self.h_s, self.topk)
            b["ws"] = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev) if ws else None
            self._bufs[n_q] = b
        return b

    def decode(self, q_idx, w, q_sfa, page_table, seq_lens, q_seq, q_pos, max_ctx, q_group=1):
        """Indexer + Top-K + SFA for n_q query rows.  Returns (out bf16 [n_q, h_s, 512],
        lse fp32 [n_q, h_s], idx int32 [n_q, topk]); the tensors are reused by the next
        call with the same n_q."""
        n_q = q_idx.shape[0]
        b = self._buffers(n_q)
        indexer_topk(q_idx, w, self.k_cache, page_table, seq_lens, q_seq, q_pos, self.topk, max_ctx,
                     q_group=q_group, out_idx=b["idx"])
        sparse_attn(q_sfa, self.kv_cache, page_table, seq_lens, q_seq, b["idx"], self.sm_scale,
                    out=b["out"], out_lse=b["lse"], workspace=b["ws"])
        return b["out"], b["lse"], b["idx"]

    def step(self, k_new, kv_new, slots_new, q_idx, w, q_sfa, page_table, seq_lens, q_seq, q_pos,
             max_ctx, q_group=1):
        """Write this step's tokens into both caches, then decode: one library call
        (dsa_decode_step).  With one new token per query row the indexer kernel writes the
        tokens itself, each before it loads the page that holds it, and SFA follows it on
        the current stream with programmatic dependent launch; otherwise a writer kernel
        runs first and the indexer reads its other inputs while the writer runs.
        """
        n_q = q_idx.shape[0]
        b = self._buffers(n_q)
        decode_step(k_new, kv_new, slots_new, self.k_cache, self.kv_cache, q_idx, w, q_sfa, page_table,
                    seq_lens, q_seq, q_pos, self.topk, max_ctx, self.sm_scale, q_group=q_group,
                    out_idx=b["idx"], out=b["out"], out_lse=b["lse"], workspace=b["ws"],
                    stream=torch.cuda.current_stream(self.device))
        return b["out"], b["lse"], b["idx"]

    def capture_step(self, inputs, max_ctx, q_group=1, stage=None, result=None):
        """Record one decode step (``step`` on the tensors of ``inputs``) into a CUDA graph
        and return a function that replays it on the current stream.

        inputs  dict with the ``step`` arguments k_new, kv_new, slots_new, q_idx, w, q_sfa,
                page_table, seq_lens, q_seq, q_pos: device tensors that stay in place; a
                replay reads whatever they hold then.
        stage   optional (pinned host tensor, device tensor) pair copied host -> device at
                the start of every replay (the step's inputs staged in one buffer).
        result  optional pinned host tensor [n_q, h_s, 512] bf16 that receives the output at
                the end of every replay.

        The graph holds the launches of one ``dsa_decode_step`` with their programmatic
        dependencies, so a replay costs one graph launch instead of the host work of each
        call.  The returned function also exposes ``out``, ``lse`` and ``idx``, the device
        tensors the replays write.
        """
        keys = ("k_new", "kv_new", "slots_new", "q_idx", "w", "q_sfa", "page_table", "seq_lens", "q_seq", "q_pos")
        args = [inputs[k] for k in keys]
        # one eager step first: per-device queries, kernel attributes and the output buffers
        # are set up outside the capture
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            if stage is not None:
                stage[1].copy_(stage[0], non_blocking=True)
            self.step(*args, max_ctx, q_group)
        torch.cuda.current_stream(self.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        # (relaxed: the library's host-side queries during the capture are not stream work)
        with torch.cuda.graph(graph, capture_error_mode="relaxed"):
            if stage is not None:
                stage[1].copy_(stage[0], non_blocking=True)
            out, lse, idx = self.step(*args, max_ctx, q_group)
            if result is not None:
                result.copy_(out, non_blocking=True)

        def replay():
            graph.replay()

        replay.out, replay.lse, replay.idx, replay.graph = out, lse, idx, graph
        return replay
