"""The benchmark's gather probes (probes.cu) read exactly the rows they name.

bench.py reports the sparse kernels against the rate at which these probes
pull row stretches named by random indices into the SMs; a probe that read
other bytes (or fewer) would give a false ceiling. Each probe's per-task
checksum (xor of every 32-bit word read, 23 low bits) is recomputed here."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_gather_probe_reads_the_named_rows(mode):
    import bench
    lib = bench.load_probes()
    F, d, rows, nnz = 300, 512 if mode in (2, 3) else 520, 37, 45
    rng = np.random.default_rng(5 + mode)
    W = rng.integers(-32768, 32767, size=(F, d), dtype=np.int16)
    idx = rng.integers(0, F, size=(rows, nnz), dtype=np.int32)
    GW = 512 if mode == 4 else 256  # columns per task
    G = (d + GW - 1) // GW
    Wd, idxd = torch.from_numpy(W).cuda(), torch.from_numpy(idx).cuda()
    sink = torch.empty(rows * G, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.probe_gather(mode, ctypes.c_void_p(Wd.data_ptr()), F, d, ctypes.c_void_p(idxd.data_ptr()), rows, nnz,
                          ctypes.c_void_p(sink.data_ptr()), ctypes.c_void_p(st.data_ptr()),
                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = sink.cpu().numpy().view(np.uint32)
    words = W.view(np.uint32).reshape(F, d // 2)
    want = np.zeros(rows * G, dtype=np.uint32)
    for r in range(rows):
        for g in range(G):
            c = words[idx[r], g * GW // 2:min((g + 1) * GW // 2, d // 2)]
            task = g * rows + r if mode == 4 else r * G + g
            want[task] = np.bitwise_xor.reduce(c.reshape(-1)) & 0x007fffff
    np.testing.assert_array_equal(got, want)


def test_fma_probe_runs():
    import bench
    peak = bench.fma_peak(torch.cuda.current_stream(), torch.cuda.get_device_properties(0).multi_processor_count)
    # 152 SMs x 128 FMA/clk x 2 FLOP at 1-2.1 GHz
    assert 20.0 < peak["fp32_fma"] < 100.0 and 20.0 < peak["bf16_mixed_fma"] < 100.0
