"""The stored container fixtures still match what the oracle writes."""
import json
import os

import numpy as np

from oracle import wcomp_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def test_fixture_matches_oracle():
    g = json.load(open(os.path.join(HERE, "golden", "containers_5x200.json")))
    w = np.frombuffer(bytes.fromhex(g["weights_hex"]), dtype="<u2").reshape(g["N"], g["K"])
    for scheme, name in ((O.BYTESPLIT, "bytesplit"), (O.K15, "k15")):
        buf = bytes.fromhex(g[name]["container_hex"])
        assert O.serialize(O.encode(w, scheme)) == buf
        c = O.deserialize(buf)
        assert c.E == g[name]["E"] > 0
        assert np.array_equal(O.decode(c), w)
