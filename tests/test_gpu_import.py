"""w4a16_pack_ex: packing from checkpoint word formats gives the same packed
buffer as w4a16_pack from the unpacked values, byte for byte.

Source words are the oracle's encodings of the same q (GPTQ sequential [N, K/8],
ExLlama [N, K/8], the MI300 [K, N/8]); scales and zero points in both the
[N][ng] and the [ng][N] orientation.
"""

import numpy as np
import pytest
import torch

import oracle as orc
from w4a16_int4_weight_gb300 import inputs as synth

from gpu_helpers import B, to_dev_bits

pytestmark = pytest.mark.gpu

SHAPES = [
    (256, 1024, 128, "uint4b8", "bf16"),
    (200, 4112, -1, "uint4b8", "fp16"),    # ragged N, K % 32 == 16
    (136, 512, 32, "uint4", "bf16"),
    (8, 16, -1, "uint4", "fp16"),          # smallest legal layer
    (1024, 768, 64, "uint4", "fp16"),
]


def _pack_buffer(p, fn):
    tot, so, zo, _ = B().packed_layout(p.N, p.K, p.group_size, p.qtype, p.dtype)
    buf = torch.zeros(tot, dtype=torch.uint8, device="cuda")   # section gaps stay zero in both
    fn(buf)
    torch.cuda.synchronize()
    return buf.cpu().numpy()


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("fmt", ["unpacked", "gptq", "exllama", "kn"])
@pytest.mark.parametrize("layout", ["ng", "gn"])
def test_import_matches_pack(sh, fmt, layout):
    N, K, G, qt, dt = sh
    if fmt == "kn" and N % 8:
        pytest.skip("the [K][N/8] format needs N % 8 == 0")
    p = synth.Problem(1, N, K, G, qt, dt)
    q, s, z = synth.make_weights(p)
    qd = torch.from_numpy(q).cuda()
    sd = to_dev_bits(s, dt)
    zd = torch.from_numpy(z).cuda() if z is not None else None
    ref = _pack_buffer(p, lambda buf: B().pack(qd, sd, zd, buf, N, K, G, qt, dt))

    src = qd if fmt == "unpacked" else torch.from_numpy(orc.encode_q(q, fmt).view(np.int32)).cuda()
    s_in = sd if layout == "ng" else to_dev_bits(np.ascontiguousarray(s.T), dt)
    z_in = None if z is None else (zd if layout == "ng" else torch.from_numpy(np.ascontiguousarray(z.T)).cuda())
    got = _pack_buffer(p, lambda buf: B().pack_ex(src, fmt, s_in, z_in, layout, buf, N, K, G, qt, dt))
    assert np.array_equal(got, ref)
