"""kv_decode_attn_noalloc: decode attention for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc (a host program linking only the C ABI
under a runtime that already owns the device's memory, or a loop that cannot take
cudaMalloc's implicit synchronisation). For them the library keeps a fixed device array in
place of the caller's workspace. This file is collected last so that a run stopping at the
first failure has already run every other test; it passes alone in a fresh process too.

Checks, through the C ABI: two calls in a row give exactly the bytes of kv_decode_attn with a
caller workspace (the same kernels and work list on the same inputs), and both agree with the
oracle's fp64 attention within the decode tolerance max(1e-3, 2e-3 |ref|); a config whose
workspace would exceed the fixed array is refused with KVQ_EUNSUPPORTED.
"""

import numpy as np
import pytest

from oracle import attention
from quantized_kv_cache_gb300 import _lib, synth

import tolerance
from gpu_cases import FAMILIES, Pair

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pair():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p = Pair(FAMILIES["kvarn4_ring"])
    p.prefill()
    yield p
    p.gpu.close()


def test_noalloc_matches_workspace_call_twice(pair):
    f = pair.f
    G = f.Hq // f.H
    for layer in range(f.L):
        q_np = np.stack([synth.q_values(f.seed, layer, s, 0, f.Hq, f.D) for s in pair.seqs])
        q = torch.from_numpy(q_np).to(pair.dev)
        ref = torch.empty_like(q)
        pair.gpu.decode_attn(layer, pair.seqs, q, ref)
        torch.cuda.synchronize()
        ref_bits = ref.cpu().numpy().view(np.uint16)
        for _ in range(2):
            out = torch.full_like(q, float("nan"))
            _lib.kv_decode_attn_noalloc(pair.gpu.h, layer, pair.seqs, q.data_ptr(), out.data_ptr())
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            assert np.array_equal(got.view(np.uint16), ref_bits), f"layer {layer}: differs from kv_decode_attn"
            for bi, s in enumerate(pair.seqs):
                for h in range(f.H):
                    hc = pair.hc[(layer, s, h)]
                    want = attention.attend(q_np[bi, h * G:(h + 1) * G].astype(np.float64), hc.regions(),
                                            hc.cfg.rot, 1.0 / np.sqrt(f.D))
                    tolerance.check(f.name + " noalloc", got[bi, h * G:(h + 1) * G], want,
                                    where=f"layer {layer} seq {s} head {h}")


def test_noalloc_refuses_workspace_beyond_fixed_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_kv_cache_gb300 import KVCache
    f = FAMILIES["kvarn5_wide"]           # D 512, 16 queries per KV head: workspace > 32 MiB
    _, ws = _lib.kv_required_bytes(f.config())
    assert ws > 32 << 20
    c = KVCache(f.config(), 0)
    try:
        dev = torch.device("cuda", 0)
        k = torch.zeros((1, 4, f.H, f.D), dtype=torch.float16, device=dev)
        c.append(0, [0], k, k)
        q = torch.zeros((1, f.Hq, f.D), dtype=torch.float16, device=dev)
        out = torch.empty_like(q)
        with pytest.raises(_lib.KVQError) as e:
            _lib.kv_decode_attn_noalloc(c.h, 0, [0], q.data_ptr(), out.data_ptr())
        assert e.value.code == 3
    finally:
        c.close()
