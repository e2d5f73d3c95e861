"""GPU parity at the edges of the accepted shapes (include/lily_moe.h): prefill
with d up to 16384 and I up to 4096, decode with d = 4096 and I = 1024, at
token counts the fp64 oracle finishes in seconds.  Same bounds as the other
parity tests: routing bit-exact, logits within the fp32 accumulation bound,
outputs within 1e-2 of the oracle's rms."""
import pytest

from bit_grouped_expert_top_gb300.inputs import CONFIGS
from test_gpu_decode import _check_decode
from test_gpu_prefill import _full_check

pytestmark = pytest.mark.gpu

TINY = CONFIGS["tiny"]


@pytest.mark.parametrize("d,I,T", [(4096, 512, 40), (8192, 256, 24), (16384, 128, 8), (2048, 2048, 32),
                                   (1024, 4096, 24)])
def test_prefill_large_shapes(d, I, T):
    # long K loops (d / 64 up to 256 k-steps), many down tiles (d / 256 up to 64),
    # many gate/up tiles (I / 128 up to 32) and down K up to 4096
    cfg = TINY.with_(d=d, I=I, I_shared=I)
    _full_check(cfg, T, seed_offset=d + I)


@pytest.mark.parametrize("T", [1, 8])
def test_decode_largest_shape(T):
    # the largest decode shape: d = 4096, I = 1024 (32 gate/up tasks per unit,
    # 8 K blocks per unit in the down projection)
    cfg = TINY.with_(d=4096, I=1024, I_shared=1024)
    _check_decode(cfg, n_layers=2, T=T)
