"""The allocation-free route + permute entry point, for callers that cannot call cudaMalloc
(plugins inside a framework that owns all device memory, code running where an allocation is
not allowed). It keeps its scratch in a static device array inside the library; this test
checks through the C ABI that it gives the same results as moe_route_permute on two calls in
a row (the second call must not see the first call's leftovers), and that it refuses sizes
beyond its fixed scratch before launching anything.

Kept in a file of its own that is collected last."""
import numpy as np
import pytest
import torch

import grouped_gemm_device_gb300 as g
from grouped_gemm_device_gb300 import synth

from .gpu_helpers import bf16_dev

pytestmark = pytest.mark.gpu


def _reference(cfg, logits, x):
    d = g.desc_from_config(cfg)
    L = g.MoELayer(d)
    L.route_permute(logits, x, cfg.T)
    torch.cuda.synchronize()
    R = L.layout.R_cap
    return (L.topk_ids.clone(), L.topk_probs.clone(), L.counts.clone(), L.offsets().clone(),
            L.ws_view("x_perm", torch.bfloat16, (R, cfg.H)).clone())


def test_noalloc_route_permute_matches_workspace_version_twice(lib):
    for cfg in (synth.LayerConfig("na1", T=700, E=64, k=4, H=256, F=64, seed=41, zipf_s=1.1),
                synth.LayerConfig("na2", T=513, E=8, k=2, H=128, F=64, seed=42),
                # 128-row segments over 256 experts: the largest padding the scratch holds
                synth.LayerConfig("na3", T=300, E=256, k=8, H=64, F=64, seed=43, zipf_s=1.1,
                                  align=128)):
        d = g.desc_from_config(cfg)
        R = cfg.T * cfg.k + cfg.E * (cfg.align - 1)
        ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
        probs = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device="cuda")
        counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
        offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda")
        x_perm = torch.full((R, cfg.H), 7.0, dtype=torch.bfloat16, device="cuda")
        for call, seed in enumerate((cfg.seed, cfg.seed + 1000)):
            c = cfg.with_(seed=seed)
            logits = torch.from_numpy(synth.gen_logits(c)).cuda()
            x = bf16_dev(synth.gen_x(c))
            want = _reference(cfg, logits, x)
            g.moe_route_permute_noalloc(d, cfg.T, logits, x, ids, probs, counts, offsets, x_perm,
                                        R)
            torch.cuda.synchronize()
            got = (ids, probs, counts, offsets, x_perm)
            for name, a, b in zip(("ids", "probs", "counts", "offsets", "x_perm"), got, want):
                if a.dtype == torch.float32:
                    assert torch.allclose(a, b, rtol=1e-6, atol=1e-7), (call, name)
                else:
                    assert torch.equal(a, b), (call, name)


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    d = g.make_desc(E=8, k=8, H=128, F=64, T_max=16385)     # 131080 pairs > 131072
    with pytest.raises(g.MoeError) as e:
        g.moe_route_permute_noalloc(d, 1, 256, 256, 256, 256, 256, 256, 256, 1 << 20)
    assert e.value.status == 2
    assert "131072" in g.load().moe_last_error_string().decode()
    # at the pair limit with 128-row segments over 256 experts the rows still fit
    d = g.make_desc(E=256, k=8, H=64, F=64, T_max=16384, align=128)
    with pytest.raises(g.MoeError) as e:
        g.moe_route_permute_noalloc(d, 1, 256, 256, 256, 256, 256, 256, 256, 1)  # x_perm short
    assert e.value.status == 1
    assert "x_perm" in g.load().moe_last_error_string().decode()
