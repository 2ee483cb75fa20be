"""liboss: online-softmax row softmax, attention forward, split-KV decode and
partial merge on one GB300 (sm_103a)."""
