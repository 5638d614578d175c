"""GB300-native DSA lightning indexer + top-k + IndexShare sparse attention."""
