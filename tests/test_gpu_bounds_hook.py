"""The bounds-checked build's checks run and are reported (svx_debug_clip_q_rows).

The hook makes the chunk launches state a smaller q than the real one; the real buffer is larger, so no
access leaves it in either build.  With libsvx_checked.so (SVX_LIBRARY=checked; this file also runs there
from tests/test_gpu_bounds_checked.py) the chunk kernel must skip the q loads past the stated extent and
raise the device error word, so the round ends in SVX_ERR_CUDA, and the next round is correct again.  With
libsvx.so the checks are compiled out and the hook changes nothing.
"""
import numpy as np
import pytest

import workloads as W
from helpers import check_parity, gpu_inputs, oracle_out, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def svx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_chunked_gb300 import svx as mod
    return mod


@pytest.mark.parametrize("resident", [True, False], ids=["resident", "streamed"])
@pytest.mark.parametrize("tensor_cores", [True, False], ids=["tc", "fma"])
def test_a_clipped_q_extent_is_caught_by_the_checked_build_only(svx, resident, tensor_cores):
    w = W.Workload("clip", 3, 16, 4, 128, (700, 129, 1500), 256, 5, seed=93)
    x, t = gpu_inputs(w, resident=resident)
    ref = oracle_out(w, x)
    checked = "bounds-checked" in svx.version()
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      tensor_cores=tensor_cores) as v:
        check_parity(*run_gpu(v, w, t, x), *ref)
        # q's last request stated as absent: its rows lie past the stated extent
        v.debug_clip_q_rows((w.n_req - 1) * w.n_q_heads * w.n_query)
        if checked:
            with pytest.raises(svx.SvxError) as e:
                run_gpu(v, w, t, x)
            assert e.value.status == svx.ERR_CUDA
            assert "outside its buffers" in str(e.value)
            site = 1 if tensor_cores else 4  # kSiteTcQ / kSiteFmaQ
            assert "0x%x" % (4 | (1 << (8 + site))) in str(e.value), str(e.value)
        else:
            check_parity(*run_gpu(v, w, t, x), *ref)
        # the hook lasts one round; the word was cleared; the next round is correct
        o, lse = run_gpu(v, w, t, x)
        check_parity(o, lse, *ref)
        assert np.all(np.isfinite(lse))
