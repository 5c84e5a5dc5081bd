"""Rotated low-bit KV cache and its decode attention for GB300 (sm_103a).

The work is done by ``lib/libkvq.so`` (hand-written CUDA behind the C ABI of
``include/kvq.h``); this package only marshals arguments (``_lib``), names the measured
workloads (``configs``), draws seeded synthetic inputs (``synth``) and wraps device memory
owned by PyTorch (``KVCache``). There is no CPU fallback: without the shared library every
call raises.
"""

from . import _lib, configs, synth  # noqa: F401
from ._lib import (KVQError, kvq_config, kv_bytes_per_token, kv_required_bytes, kv_create,  # noqa: F401
                   kv_destroy, kv_reset, kv_append, kv_prefill, kv_seal, kv_decode_attn, kv_state, kv_get_status,
                   kv_dequant, kv_region_ptr, kv_format_tables, kvq_synth_fill)


class KVCache:
    """A cache whose device pool and decode workspace are PyTorch CUDA tensors."""

    def __init__(self, cfg, device=0):
        import torch
        self.cfg = cfg
        self.device = device
        self.pool_bytes, self.ws_bytes = kv_required_bytes(cfg)
        dev = torch.device("cuda", device)
        self.pool = torch.empty(self.pool_bytes, dtype=torch.uint8, device=dev)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        with torch.cuda.device(dev):
            self.h = kv_create(cfg, self.pool.data_ptr(), self.pool_bytes, device)

    def close(self):
        if self.h is not None:
            kv_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def append(self, layer, seq_ids, k, v, stream=0):
        """k, v: fp16 CUDA tensors [n_seq, n_tok, H, D] (contiguous)."""
        assert k.is_contiguous() and v.is_contiguous()
        kv_append(self.h, layer, seq_ids, k.shape[1], k.data_ptr(), v.data_ptr(), stream)

    def prefill(self, layer, seq_ids, k, v, keep, stream=0):
        """kv_prefill: k, v fp16 CUDA tensors [n_seq, n_tok, H, D] (contiguous). Returns the
        number of groups sealed."""
        assert k.is_contiguous() and v.is_contiguous()
        return kv_prefill(self.h, layer, seq_ids, k.shape[1], k.data_ptr(), v.data_ptr(), keep, stream)

    def seal(self, layer, seq_ids, keep, stream=0):
        return kv_seal(self.h, layer, seq_ids, keep, stream)

    def decode_attn(self, layer, seq_ids, q, out, stream=0):
        """q, out: fp16 CUDA tensors [n_seq, Hq, D] (contiguous)."""
        assert q.is_contiguous() and out.is_contiguous()
        kv_decode_attn(self.h, layer, seq_ids, q.data_ptr(), out.data_ptr(), self.ws.data_ptr(), self.ws_bytes,
                       stream)

    def state(self, layer, seq):
        return kv_state(self.h, layer, seq)
