"""The codebook file (.fqb): the codec's persistent state round-trips bit for bit, and a damaged
file is refused rather than loaded."""
import numpy as np
import pytest

from random_access_kv_gb300 import codebook as pcb


def _tables():
    r = np.random.default_rng(3)
    return r.standard_normal((256, 2)).astype(np.float32), pcb.haar(r.standard_normal((64, 64))).astype(np.float32)


def test_round_trip(tmp_path):
    C, Pi = _tables()
    p = tmp_path / "w2.fqb"
    pcb.save_fqb(str(p), C, Pi, "spiral", seed=2, iters=20, restarts=4, draws=65536, mse=2.29e-4)
    C2, Pi2, meta = pcb.load_fqb(str(p))
    assert C2.tobytes() == C.tobytes() and Pi2.tobytes() == Pi.tobytes()
    assert meta == {"d": 64, "k": 2, "N": 256, "kind": "spiral", "seed": 2, "lloyd_iters": 20, "restarts": 4,
                    "draws": 65536, "mse": 2.29e-4}


@pytest.mark.parametrize("damage", ["flip", "truncate", "magic", "extend"])
def test_damaged_files_are_refused(tmp_path, damage):
    C, Pi = _tables()
    p = tmp_path / "x.fqb"
    pcb.save_fqb(str(p), C, Pi, "spiral")
    b = bytearray(p.read_bytes())
    if damage == "flip":
        b[100] ^= 0x10
    elif damage == "truncate":
        b = b[:-9]
    elif damage == "magic":
        b[0:4] = b"XXXX"
    else:
        b += b"\0"
    p.write_bytes(bytes(b))
    with pytest.raises(ValueError):
        pcb.load_fqb(str(p))
